/* _fastcall.c -- CPython entry points for the per-step calls of libqsa.so.
 *
 * Marshalling only, like the ctypes path it stands in for: each function
 * takes the C function's arguments in order (device pointers as Python ints
 * or None, sizes as ints, the RoPE base as a float), calls the library and
 * returns its status.  It exists because a ctypes call converts its
 * arguments one by one through their declared types (about 0.13 us each on
 * the host, 26 of them per decode step), which is a large share of a decode
 * step's host time.  The Python module falls back to ctypes when this
 * extension was not built.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include "qsa.h"

/* Argument i as a pointer (None -> NULL), a 64-bit or 32-bit integer, a
 * size or a double; any failure leaves a Python error set. */
static void* arg_ptr(PyObject* const* a, Py_ssize_t i) {
  if (a[i] == Py_None) return NULL;
  return PyLong_AsVoidPtr(a[i]);
}
static int64_t arg_i64(PyObject* const* a, Py_ssize_t i) { return (int64_t)PyLong_AsLongLong(a[i]); }
static int32_t arg_i32(PyObject* const* a, Py_ssize_t i) {
  const long long v = PyLong_AsLongLong(a[i]);
  if (!PyErr_Occurred() && (v < INT32_MIN || v > INT32_MAX)) PyErr_SetString(PyExc_OverflowError, "int32 argument");
  return (int32_t)v;
}
static size_t arg_size(PyObject* const* a, Py_ssize_t i) { return (size_t)PyLong_AsSize_t(a[i]); }

static int want_args(Py_ssize_t got, Py_ssize_t n, const char* fn) {
  if (got == n) return 1;
  PyErr_Format(PyExc_TypeError, "%s takes %zd arguments (%zd given)", fn, n, got);
  return 0;
}

/* qsa_decode_step and qsa_decode_step_gated share every argument but the
 * gates (after q). */
static PyObject* decode_step_impl(PyObject* const* a, Py_ssize_t n, int gated) {
  const Py_ssize_t g = gated ? 1 : 0;
  if (!want_args(n, 26 + g, gated ? "decode_step_gated" : "decode_step")) return NULL;
  const void* new_keys = arg_ptr(a, 0);
  const int32_t* req_tok_start = arg_ptr(a, 1);
  const int32_t* req_first_pos = arg_ptr(a, 2);
  void* ring = arg_ptr(a, 3);
  const double rope_base = PyFloat_AsDouble(a[4]);
  const void* q = arg_ptr(a, 5);
  const float* gates = gated ? (const float*)arg_ptr(a, 6) : NULL;
  void* pool = arg_ptr(a, 6 + g);
  const int64_t pool_rows = arg_i64(a, 7 + g);
  const int32_t n_req = arg_i32(a, 8 + g);
  const int32_t* req_row_start = arg_ptr(a, 9 + g);
  const int32_t n_rows = arg_i32(a, 10 + g);
  const int32_t* row_len = arg_ptr(a, 11 + g);
  const int32_t max_len = arg_i32(a, 12 + g), max_rows_per_req = arg_i32(a, 13 + g);
  const int32_t* page_table = arg_ptr(a, 14 + g);
  const int64_t ld_pt = arg_i64(a, 15 + g);
  const int32_t page_size = arg_i32(a, 16 + g), k_blk = arg_i32(a, 17 + g);
  int32_t* out_blocks = arg_ptr(a, 18 + g);
  int32_t* out_pos = arg_ptr(a, 19 + g);
  int32_t* out_slots = arg_ptr(a, 20 + g);
  float* scores_out = arg_ptr(a, 21 + g);
  const int64_t ld_scores = arg_i64(a, 22 + g);
  void* workspace = arg_ptr(a, 23 + g);
  const size_t ws_bytes = arg_size(a, 24 + g);
  void* stream = arg_ptr(a, 25 + g);
  if (PyErr_Occurred()) return NULL;
  const qsa_status st =
      gated ? qsa_decode_step_gated(new_keys, req_tok_start, req_first_pos, ring, rope_base, q, gates, pool,
                                    pool_rows, n_req, req_row_start, n_rows, row_len, max_len, max_rows_per_req,
                                    page_table, ld_pt, page_size, k_blk, out_blocks, out_pos, out_slots,
                                    scores_out, ld_scores, workspace, ws_bytes, stream)
            : qsa_decode_step(new_keys, req_tok_start, req_first_pos, ring, rope_base, q, pool, pool_rows, n_req,
                              req_row_start, n_rows, row_len, max_len, max_rows_per_req, page_table, ld_pt,
                              page_size, k_blk, out_blocks, out_pos, out_slots, scores_out, ld_scores, workspace,
                              ws_bytes, stream);
  return PyLong_FromLong((long)st);
}

static PyObject* fc_decode_step(PyObject* self, PyObject* const* a, Py_ssize_t n) {
  (void)self;
  return decode_step_impl(a, n, 0);
}
static PyObject* fc_decode_step_gated(PyObject* self, PyObject* const* a, Py_ssize_t n) {
  (void)self;
  return decode_step_impl(a, n, 1);
}

/* qsa_indexer_select (pool) and qsa_indexer_select_gated (gates, pool). */
static PyObject* indexer_select_impl(PyObject* const* a, Py_ssize_t n, int gated) {
  const Py_ssize_t g = gated ? 1 : 0;
  if (!want_args(n, 21 + g, gated ? "indexer_select_gated" : "indexer_select")) return NULL;
  const void* q = arg_ptr(a, 0);
  const float* gates = gated ? (const float*)arg_ptr(a, 1) : NULL;
  const void* pool = arg_ptr(a, 1 + g);
  const int64_t pool_rows = arg_i64(a, 2 + g);
  const int32_t n_req = arg_i32(a, 3 + g);
  const int32_t* req_row_start = arg_ptr(a, 4 + g);
  const int32_t n_rows = arg_i32(a, 5 + g);
  const int32_t* row_len = arg_ptr(a, 6 + g);
  const int32_t max_len = arg_i32(a, 7 + g), max_rows_per_req = arg_i32(a, 8 + g);
  const int32_t* page_table = arg_ptr(a, 9 + g);
  const int64_t ld_pt = arg_i64(a, 10 + g);
  const int32_t page_size = arg_i32(a, 11 + g), k_blk = arg_i32(a, 12 + g);
  int32_t* out_blocks = arg_ptr(a, 13 + g);
  int32_t* out_pos = arg_ptr(a, 14 + g);
  int32_t* out_slots = arg_ptr(a, 15 + g);
  float* scores_out = arg_ptr(a, 16 + g);
  const int64_t ld_scores = arg_i64(a, 17 + g);
  void* workspace = arg_ptr(a, 18 + g);
  const size_t ws_bytes = arg_size(a, 19 + g);
  void* stream = arg_ptr(a, 20 + g);
  if (PyErr_Occurred()) return NULL;
  const qsa_status st =
      gated ? qsa_indexer_select_gated(q, gates, pool, pool_rows, n_req, req_row_start, n_rows, row_len, max_len,
                                       max_rows_per_req, page_table, ld_pt, page_size, k_blk, out_blocks, out_pos,
                                       out_slots, scores_out, ld_scores, workspace, ws_bytes, stream)
            : qsa_indexer_select(q, pool, pool_rows, n_req, req_row_start, n_rows, row_len, max_len,
                                 max_rows_per_req, page_table, ld_pt, page_size, k_blk, out_blocks, out_pos,
                                 out_slots, scores_out, ld_scores, workspace, ws_bytes, stream);
  return PyLong_FromLong((long)st);
}

static PyObject* fc_indexer_select(PyObject* self, PyObject* const* a, Py_ssize_t n) {
  (void)self;
  return indexer_select_impl(a, n, 0);
}
static PyObject* fc_indexer_select_gated(PyObject* self, PyObject* const* a, Py_ssize_t n) {
  (void)self;
  return indexer_select_impl(a, n, 1);
}

static PyMethodDef fc_methods[] = {
    {"qsa_decode_step", (PyCFunction)(void (*)(void))fc_decode_step, METH_FASTCALL, "qsa_decode_step"},
    {"qsa_decode_step_gated", (PyCFunction)(void (*)(void))fc_decode_step_gated, METH_FASTCALL,
     "qsa_decode_step_gated"},
    {"qsa_indexer_select", (PyCFunction)(void (*)(void))fc_indexer_select, METH_FASTCALL, "qsa_indexer_select"},
    {"qsa_indexer_select_gated", (PyCFunction)(void (*)(void))fc_indexer_select_gated, METH_FASTCALL,
     "qsa_indexer_select_gated"},
    {NULL, NULL, 0, NULL}};

static struct PyModuleDef fc_module = {PyModuleDef_HEAD_INIT,
                                       "_fastcall",
                                       "Per-step calls of libqsa.so without ctypes argument conversion.",
                                       -1,
                                       fc_methods,
                                       NULL,
                                       NULL,
                                       NULL,
                                       NULL};

PyMODINIT_FUNC PyInit__fastcall(void) { return PyModule_Create(&fc_module); }
