/*
 * pycalls.c -- the CPython extension `_calls`: argument conversion for the
 * five entry points of libattn that launch kernels (attn_prefill_causal,
 * attn_decode, attn_decode_append, attn_decode_noalloc, kv_append).
 *
 * A decode step is a few microseconds of GPU work, and a ctypes call with
 * 15-19 converted arguments costs a noticeable share of that on the host.
 * This module does the same marshalling in C: every buffer argument is None
 * (NULL), an int (a raw address) or an object with a data_ptr() method (a
 * torch tensor); sizes are non-negative ints below 2^32 (anything else
 * raises OverflowError or TypeError before the library is called); the
 * stream is an int (a cudaStream_t) or an object with a `cuda_stream`
 * attribute.  It computes nothing.
 *
 * The module is not linked against libattn.so: the Python package loads the
 * library once and hands this module the addresses of its functions
 * (bind()), so both bindings call into the same loaded copy.  The GIL is
 * released while the library runs.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include <stdint.h>

#include "../../include/attn.h"

static __typeof__(&attn_prefill_causal) p_prefill_causal;
static __typeof__(&attn_decode) p_decode;
static __typeof__(&attn_decode_append) p_decode_append;
static __typeof__(&attn_decode_noalloc) p_decode_noalloc;
static __typeof__(&kv_append) p_kv_append;

static PyObject* s_data_ptr;     /* interned "data_ptr" */
static PyObject* s_cuda_stream;  /* interned "cuda_stream" */

static int long_to_addr(PyObject* v, void** out) {
    const unsigned long long x = PyLong_AsUnsignedLongLong(v);
    if (x == (unsigned long long)-1 && PyErr_Occurred()) return -1;
    *out = (void*)(uintptr_t)x;
    return 0;
}

/* None -> NULL; int -> that address; otherwise obj.data_ptr(). */
static int as_ptr(PyObject* o, void** out) {
    if (o == Py_None) {
        *out = NULL;
        return 0;
    }
    if (PyLong_Check(o)) return long_to_addr(o, out);
    PyObject* v = PyObject_CallMethodNoArgs(o, s_data_ptr);
    if (!v) return -1;
    const int r = PyLong_Check(v) ? long_to_addr(v, out)
                                  : (PyErr_SetString(PyExc_TypeError, "data_ptr() is not an int"), -1);
    Py_DECREF(v);
    return r;
}

/* int -> that cudaStream_t; otherwise obj.cuda_stream. */
static int as_stream(PyObject* o, void** out) {
    if (PyLong_Check(o)) return long_to_addr(o, out);
    PyObject* v = PyObject_GetAttr(o, s_cuda_stream);
    if (!v) return -1;
    const int r = PyLong_Check(v) ? long_to_addr(v, out)
                                  : (PyErr_SetString(PyExc_TypeError, "cuda_stream is not an int"), -1);
    Py_DECREF(v);
    return r;
}

static int as_u64(PyObject* o, unsigned long long* out) {
    PyObject* i = PyNumber_Index(o);
    if (!i) return -1;
    const unsigned long long x = PyLong_AsUnsignedLongLong(i);
    Py_DECREF(i);
    if (x == (unsigned long long)-1 && PyErr_Occurred()) return -1;
    *out = x;
    return 0;
}

static int as_u32(PyObject* o, uint32_t* out) {
    unsigned long long x;
    if (as_u64(o, &x)) return -1;
    if (x > 0xffffffffull) {
        PyErr_SetString(PyExc_OverflowError, "size argument does not fit in 32 bits");
        return -1;
    }
    *out = (uint32_t)x;
    return 0;
}

static int as_size(PyObject* o, size_t* out) {
    unsigned long long x;
    if (as_u64(o, &x)) return -1;
    *out = (size_t)x;
    return 0;
}

static int as_f32(PyObject* o, float* out) {
    const double x = PyFloat_AsDouble(o);
    if (x == -1.0 && PyErr_Occurred()) return -1;
    *out = (float)x;
    return 0;
}

static int as_int(PyObject* o, int* out) {
    PyObject* i = PyNumber_Index(o);
    if (!i) return -1;
    const long x = PyLong_AsLong(i);
    Py_DECREF(i);
    if (x == -1 && PyErr_Occurred()) return -1;
    if (x < INT32_MIN || x > INT32_MAX) {
        PyErr_SetString(PyExc_OverflowError, "precision does not fit in an int");
        return -1;
    }
    *out = (int)x;
    return 0;
}

static int check_nargs(const char* name, Py_ssize_t nargs, Py_ssize_t want) {
    if (nargs == want) return 0;
    PyErr_Format(PyExc_TypeError, "%s takes %zd positional arguments (%zd given)", name, want,
                 nargs);
    return -1;
}

static int check_bound(void) {
    if (p_prefill_causal) return 0;
    PyErr_SetString(PyExc_RuntimeError, "_calls.bind() has not been called");
    return -1;
}

/* attn_prefill_causal(q, k, v, o, m, num_q_heads, num_kv_heads, head_dim,
 *                     q_stride, kv_stride, scale, precision, workspace,
 *                     workspace_bytes, stream) -> status */
static PyObject* py_prefill_causal(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    void *q, *k, *v, *o, *ws, *st;
    uint32_t m, hq, hkv, d, qs, kvs;
    float scale;
    int prec;
    size_t wsb;
    if (check_bound() || check_nargs("attn_prefill_causal", n, 15) || as_ptr(a[0], &q) ||
        as_ptr(a[1], &k) || as_ptr(a[2], &v) || as_ptr(a[3], &o) || as_u32(a[4], &m) ||
        as_u32(a[5], &hq) || as_u32(a[6], &hkv) || as_u32(a[7], &d) || as_u32(a[8], &qs) ||
        as_u32(a[9], &kvs) || as_f32(a[10], &scale) || as_int(a[11], &prec) ||
        as_ptr(a[12], &ws) || as_size(a[13], &wsb) || as_stream(a[14], &st))
        return NULL;
    attn_status_t r;
    Py_BEGIN_ALLOW_THREADS
    r = p_prefill_causal((const float*)q, (const float*)k, (const float*)v, (float*)o, m, hq, hkv,
                         d, qs, kvs, scale, (attn_precision_t)prec, ws, wsb, st);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong((long)r);
}

/* attn_decode(q, k_cache, v_cache, out, num_heads, kv_heads, head_dim,
 *             max_seq, total_seq, window, scale, workspace, workspace_bytes,
 *             stream) -> status */
static PyObject* py_decode(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    void *q, *kc, *vc, *out, *ws, *st;
    uint32_t hq, hkv, d, S, T, W;
    float scale;
    size_t wsb;
    if (check_bound() || check_nargs("attn_decode", n, 14) || as_ptr(a[0], &q) ||
        as_ptr(a[1], &kc) || as_ptr(a[2], &vc) || as_ptr(a[3], &out) || as_u32(a[4], &hq) ||
        as_u32(a[5], &hkv) || as_u32(a[6], &d) || as_u32(a[7], &S) || as_u32(a[8], &T) ||
        as_u32(a[9], &W) || as_f32(a[10], &scale) || as_ptr(a[11], &ws) ||
        as_size(a[12], &wsb) || as_stream(a[13], &st))
        return NULL;
    attn_status_t r;
    Py_BEGIN_ALLOW_THREADS
    r = p_decode((const float*)q, (const float*)kc, (const float*)vc, (float*)out, hq, hkv, d, S,
                 T, W, scale, ws, wsb, st);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong((long)r);
}

/* attn_decode_append(q, k_new, v_new, rope_cos, rope_sin, k_cache, v_cache,
 *                    out, num_heads, kv_heads, head_dim, max_seq, total_seq,
 *                    position, window, scale, workspace, workspace_bytes,
 *                    stream) -> status */
static PyObject* py_decode_append(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    void *q, *kn, *vn, *cs, *sn, *kc, *vc, *out, *ws, *st;
    uint32_t hq, hkv, d, S, T, pos, W;
    float scale;
    size_t wsb;
    if (check_bound() || check_nargs("attn_decode_append", n, 19) || as_ptr(a[0], &q) ||
        as_ptr(a[1], &kn) || as_ptr(a[2], &vn) || as_ptr(a[3], &cs) || as_ptr(a[4], &sn) ||
        as_ptr(a[5], &kc) || as_ptr(a[6], &vc) || as_ptr(a[7], &out) || as_u32(a[8], &hq) ||
        as_u32(a[9], &hkv) || as_u32(a[10], &d) || as_u32(a[11], &S) || as_u32(a[12], &T) ||
        as_u32(a[13], &pos) || as_u32(a[14], &W) || as_f32(a[15], &scale) ||
        as_ptr(a[16], &ws) || as_size(a[17], &wsb) || as_stream(a[18], &st))
        return NULL;
    attn_status_t r;
    Py_BEGIN_ALLOW_THREADS
    r = p_decode_append((const float*)q, (const float*)kn, (const float*)vn, (const float*)cs,
                        (const float*)sn, (float*)kc, (float*)vc, (float*)out, hq, hkv, d, S, T,
                        pos, W, scale, ws, wsb, st);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong((long)r);
}

/* attn_decode_noalloc(q, k_cache, v_cache, out, num_heads, kv_heads,
 *                     head_dim, max_seq, total_seq, window, scale, stream)
 *                     -> status */
static PyObject* py_decode_noalloc(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    void *q, *kc, *vc, *out, *st;
    uint32_t hq, hkv, d, S, T, W;
    float scale;
    if (check_bound() || check_nargs("attn_decode_noalloc", n, 12) || as_ptr(a[0], &q) ||
        as_ptr(a[1], &kc) || as_ptr(a[2], &vc) || as_ptr(a[3], &out) || as_u32(a[4], &hq) ||
        as_u32(a[5], &hkv) || as_u32(a[6], &d) || as_u32(a[7], &S) || as_u32(a[8], &T) ||
        as_u32(a[9], &W) || as_f32(a[10], &scale) || as_stream(a[11], &st))
        return NULL;
    attn_status_t r;
    Py_BEGIN_ALLOW_THREADS
    r = p_decode_noalloc((const float*)q, (const float*)kc, (const float*)vc, (float*)out, hq, hkv,
                         d, S, T, W, scale, st);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong((long)r);
}

/* kv_append(k_src, v_src, k_cache, v_cache, kv_heads, head_dim, max_seq,
 *           position, stream) -> status */
static PyObject* py_kv_append(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    void *ks, *vs, *kc, *vc, *st;
    uint32_t hkv, d, S, pos;
    if (check_bound() || check_nargs("kv_append", n, 9) || as_ptr(a[0], &ks) ||
        as_ptr(a[1], &vs) || as_ptr(a[2], &kc) || as_ptr(a[3], &vc) || as_u32(a[4], &hkv) ||
        as_u32(a[5], &d) || as_u32(a[6], &S) || as_u32(a[7], &pos) || as_stream(a[8], &st))
        return NULL;
    attn_status_t r;
    Py_BEGIN_ALLOW_THREADS
    r = p_kv_append((const float*)ks, (const float*)vs, (float*)kc, (float*)vc, hkv, d, S, pos, st);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong((long)r);
}

/* bind(prefill_causal, decode, decode_append, decode_noalloc, kv_append):
 * the addresses of those libattn functions, as ints. */
static PyObject* py_bind(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    void* f[5];
    if (check_nargs("bind", n, 5)) return NULL;
    for (int i = 0; i < 5; ++i) {
        if (!PyLong_Check(a[i])) {
            PyErr_SetString(PyExc_TypeError, "bind() takes function addresses as ints");
            return NULL;
        }
        if (long_to_addr(a[i], &f[i])) return NULL;
        if (!f[i]) {
            PyErr_SetString(PyExc_ValueError, "bind(): null function address");
            return NULL;
        }
    }
    p_prefill_causal = (__typeof__(p_prefill_causal))f[0];
    p_decode = (__typeof__(p_decode))f[1];
    p_decode_append = (__typeof__(p_decode_append))f[2];
    p_decode_noalloc = (__typeof__(p_decode_noalloc))f[3];
    p_kv_append = (__typeof__(p_kv_append))f[4];
    Py_RETURN_NONE;
}

static PyMethodDef methods[] = {
    {"bind", (PyCFunction)(void (*)(void))py_bind, METH_FASTCALL, NULL},
    {"attn_prefill_causal", (PyCFunction)(void (*)(void))py_prefill_causal, METH_FASTCALL, NULL},
    {"attn_decode", (PyCFunction)(void (*)(void))py_decode, METH_FASTCALL, NULL},
    {"attn_decode_append", (PyCFunction)(void (*)(void))py_decode_append, METH_FASTCALL, NULL},
    {"attn_decode_noalloc", (PyCFunction)(void (*)(void))py_decode_noalloc, METH_FASTCALL, NULL},
    {"kv_append", (PyCFunction)(void (*)(void))py_kv_append, METH_FASTCALL, NULL},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_calls", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__calls(void) {
    s_data_ptr = PyUnicode_InternFromString("data_ptr");
    s_cuda_stream = PyUnicode_InternFromString("cuda_stream");
    if (!s_data_ptr || !s_cuda_stream) return NULL;
    return PyModule_Create(&module);
}
