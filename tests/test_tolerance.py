"""The sparse-attention parity bound against FP32 evaluations in the
kernel's order (CPU only).

`gpu_util.attn_tolerance` is derived from the kernel's arithmetic. Each
logit is a tensor-core FP32 accumulation of exact BF16 products, in D/16
steps of 16. The weights come from exp in FP32, and every warp adds its
weighted rows in order. These tests evaluate the same attention in
numpy float32, in that order and with truncating steps, and check that the
bound holds against the FP64 oracle. They also check that the bound stays
well below the values it guards."""
import numpy as np
import pytest

import oracle
from gpu_util import attn_tolerance

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    u = x.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _truncate(x):
    """Round a float32 array towards zero to 23 fraction bits minus one (an
    adder that drops a guard bit)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    return (u & np.uint32(0xFFFFFFFE)).view(np.float32)


def _fp32_attention(q, k, v, slots, scale, truncating):
    """float32 attention in the kernel's order: logits as D/16 steps of 16
    products added to an FP32 accumulator, weights exp(logit - max), value
    sums over the chunk's rows in order, then the division."""
    qf, kf, vf = _f32(q), _f32(k), _f32(v)
    rows, h_q, d = qf.shape
    g = h_q // kf.shape[1]
    out = np.zeros((rows, h_q, d), np.float32)
    for t in range(rows):
        sl = slots[t]
        ok = sl >= 0
        for h in range(h_q):
            kk = kf[np.where(ok, sl, 0), h // g]            # [n][d]
            prod = (kk * qf[t, h]).astype(np.float32)       # exact for BF16 x BF16
            acc = np.zeros(sl.size, np.float32)
            for s in range(d // 16):
                step = prod[:, 16 * s:16 * s + 16].sum(axis=1, dtype=np.float32)
                acc = (acc + step).astype(np.float32)
                if truncating:
                    acc = _truncate(acc)
            logit = np.where(ok, np.float32(scale) * acc, -np.inf).astype(np.float32)
            if not ok.any():
                continue
            m = logit.max()
            w = np.where(ok, np.exp((logit - m).astype(np.float32)), 0).astype(np.float32)
            lsum = np.float32(0)
            o = np.zeros(d, np.float32)
            for j in range(sl.size):
                if ok[j]:
                    lsum = np.float32(lsum + w[j])
                    o = (o + w[j] * vf[sl[j], h // g]).astype(np.float32)
            out[t, h] = o / lsum
    return out


@pytest.mark.parametrize("truncating", [False, True])
@pytest.mark.parametrize("h_q,h_kv,d", [(16, 2, 256), (16, 1, 128)])
def test_attention_bound_covers_fp32_in_kernel_order(truncating, h_q, h_kv, d):
    rng = np.random.default_rng(h_q + h_kv + d + int(truncating))
    n_slots, rows, n = 700, 3, 300
    q = _bf16(rng, (rows, h_q, d))
    k = _bf16(rng, (n_slots, h_kv, d))
    v = _bf16(rng, (n_slots, h_kv, d))
    slots = rng.integers(0, n_slots, size=(rows, n)).astype(np.int32)
    slots[0, rng.random(n) < 0.3] = -1
    slots[2, 1:] = -1  # a single entry
    scale = d ** -0.5
    ref, _, _ = oracle.sparse_attn(q, k, v, slots, scale)
    got = _fp32_attention(q, k, v, slots, scale, truncating)
    tol = attn_tolerance(q, k, v, slots, scale)
    err = np.abs(got.astype(np.float64) - ref)
    assert (err <= tol).all(), float((err / tol).max())
    # and the bound is tight enough to catch a wrong head, slot or scale
    vmax = np.abs(_f32(v)).max()
    assert tol.max() < 2e-3 * vmax
