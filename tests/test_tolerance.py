"""Parity bounds against FP32 evaluations in the kernels' order (CPU only).

Compressed keys: `gpu_util.key_tolerance` (one BF16 ulp plus an absolute
term for the FP32 rotation) against the key path evaluated in numpy float32
in the kernel's order (token-order sum, fused multiply-add norm, 8-lane
butterfly, reciprocal square root, angle from the 64-bit turn fraction,
rotation with and without a fused multiply-add), on keys of the 32-request
batch up to 131K tokens.

Sparse attention:
`gpu_util.attn_tolerance` is derived from the kernel's arithmetic. Each
logit is a tensor-core FP32 accumulation of exact BF16 products, in D/16
steps of 16. The weights come from exp in FP32, and every warp adds its
weighted rows in order. These tests evaluate the same attention in
numpy float32, in that order and with truncating steps, and check that the
bound holds against the FP64 oracle. They also check that the bound stays
well below the values it guards."""
import numpy as np
import pytest

import math

import oracle
from gpu_util import KEY_ABS_TERM, attn_tolerance, key_tolerance

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


# ----------------------------------------------------------------- compressed keys
def _rope_turns(base):
    """Per frequency i, base^(-2i/128) / (2 pi) as a 64-bit fraction of a turn
    (the host computes these in FP64 and passes them to the kernel)."""
    return [(int(round(math.ldexp(base ** (-2.0 * i / 128) / (2 * math.pi), 62))) << 2) & (2 ** 64 - 1)
            for i in range(64)]


def _fma32(a, b, c):
    """FP32 fused multiply-add (the product is exact in FP64)."""
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def _bf16_rne(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _fp32_compress(raw4, pos, turns, order):
    """One compressed key in float32, in the kernel's order.  order 0: the
    rotation as plain products and a difference; 1 and 2: one product fused
    into the difference (either way a compiler may contract it)."""
    f32 = np.float32
    k = _f32(raw4)
    m = (((k[0] + k[1]) + k[2]) + k[3]) * f32(0.25)
    lo, hi = m[:64], m[64:]
    part = []
    for j in range(8):  # lane j: dims [8j, 8j+8) and [64+8j, 64+8j+8)
        s = f32(0)
        for e in range(8):
            s = _fma32(lo[8 * j + e], lo[8 * j + e], s)
            s = _fma32(hi[8 * j + e], hi[8 * j + e], s)
        part.append(s)
    ss = f32(f32(f32(part[0] + part[1]) + f32(part[2] + part[3])) + f32(f32(part[4] + part[5]) +
                                                                       f32(part[6] + part[7])))
    inv = f32(1) / np.sqrt(ss) if ss > 0 else f32(0)
    out = np.zeros(128, np.float32)
    for i in range(64):
        top = ((pos * turns[i]) & (2 ** 64 - 1)) >> 32
        top = top - 2 ** 32 if top >= 2 ** 31 else top
        y = f32(f32(top) * f32(2.0 ** -31))  # angle in units of pi
        sn, cs = f32(math.sin(math.pi * float(y))), f32(math.cos(math.pi * float(y)))
        u, v = f32(lo[i] * inv), f32(hi[i] * inv)
        if order == 0:
            a, b = f32(f32(u * cs) - f32(v * sn)), f32(f32(v * cs) + f32(u * sn))
        elif order == 1:
            a, b = _fma32(u, cs, -f32(v * sn)), _fma32(v, cs, f32(u * sn))
        else:
            a, b = _fma32(-v, sn, f32(u * cs)), _fma32(u, sn, f32(v * cs))
        out[i], out[64 + i] = a, b
    return _bf16_rne(out)


def test_compressed_key_bound_covers_the_fp32_key_path():
    """Every element of 800 keys of the 32-request batch (positions up to
    131K tokens), in three evaluation orders, is within key_tolerance of the
    FP64 oracle; without the absolute term some are not (near-cancelling
    rotations, where the result's BF16 ulp is below the FP32 error)."""
    from workloads import c3_batched
    w = c3_batched(0)
    turns = _rope_turns(w.rope_base)
    rng = np.random.default_rng(17)
    over_ulp = 0
    for i in rng.choice(w.n_blocks, 800, replace=False):
        b = int(w.block_id[i])
        raw4 = w.raw_keys[4 * i: 4 * i + 4]
        want = oracle.bf16_to_float(oracle.compress_block(raw4, 4 * b, w.rope_base))
        for order in range(3):
            got = oracle.bf16_to_float(_fp32_compress(raw4, 4 * b, turns, order))
            err = np.abs(got - want)
            tol = key_tolerance(got, want)
            assert (err <= tol).all(), (int(i), order, float((err - tol).max()))
            over_ulp += int((err > tol - KEY_ABS_TERM).sum())
    # the absolute term is needed: some elements exceed one ulp alone
    assert over_ulp > 0
