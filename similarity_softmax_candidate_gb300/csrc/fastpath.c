/*
 * _fastpath: the per-call argument marshalling of the Python binding for the
 * two readout calls, in C.
 *
 * The binding's job on every call is to check the tensors (CUDA, dtype,
 * shape, contiguity, one device, the current one), take their data
 * pointers, find the stream and call the library. Done with ctypes that
 * costs about 4 us, more than the kernel of a single question; done here,
 * with the same checks made through the same tensor attributes, it costs
 * well under 1 us. Nothing here computes anything of the readout: every
 * step runs in the library's kernels, reached through function pointers the
 * binding hands over from its ctypes handle, so this module links neither
 * the library nor CUDA.
 *
 * score(q, C, out, normalize, scale, temperature, stream, c_bf16) and
 * score_batch(Q, C, out, ...) return the library's status as an int, or
 * None when the arguments are not the plain case (a CPU tensor, a wrong
 * dtype or shape, a non-contiguous tensor, tensors on another device than
 * the current one, an unusual stream object): the binding then takes its
 * ctypes path, which raises the precise error or switches devices. c_bf16
 * says which entry point is meant: C float32 (0) or bfloat16 (1).
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>

typedef int (*score1_fn)(const void*, const void*, int, int, int, float, float, void*, void*);
typedef int (*scoreb_fn)(const void*, const void*, int, int, int, int, float, float, void*, void*);

static score1_fn g_single[2];  /* [C is bfloat16] */
static scoreb_fn g_batch[2];
static PyObject *g_f32, *g_bf16;           /* torch.float32, torch.bfloat16 */
static PyObject *g_cur_device;             /* () -> int: the current CUDA device */
static PyObject *g_raw_stream;             /* (device) -> int: its current raw stream */
static PyObject *s_is_cuda, *s_dtype, *s_shape, *s_is_contiguous, *s_data_ptr, *s_get_device, *s_cuda_stream;

/* Facts of one tensor: data pointer, device, its shape (up to 3 dims).
 * Returns 1 when it is a contiguous CUDA tensor of `ndim` dims of dtype
 * float32 (bf16 = 0) or bfloat16 (bf16 = 1), 0 otherwise (and on any
 * Python error, which is cleared). */
static int facts(PyObject* t, int ndim, int bf16, void** ptr, long* dev, long long* shape) {
    int ok = 0;
    PyObject *v = NULL, *sh = NULL;
    v = PyObject_GetAttr(t, s_is_cuda);
    if (v != Py_True) goto done;
    Py_DECREF(v);
    v = PyObject_GetAttr(t, s_dtype);
    if (!v || v != (bf16 ? g_bf16 : g_f32)) goto done;
    Py_DECREF(v);
    v = NULL;
    sh = PyObject_GetAttr(t, s_shape);
    if (!sh || !PyTuple_Check(sh) || PyTuple_GET_SIZE(sh) != ndim) goto done;
    for (int i = 0; i < ndim; ++i) {
        shape[i] = PyLong_AsLongLong(PyTuple_GET_ITEM(sh, i));
        if (shape[i] == -1 && PyErr_Occurred()) goto done;
    }
    PyObject* self[1] = {t};
    v = PyObject_VectorcallMethod(s_is_contiguous, self, 1 | PY_VECTORCALL_ARGUMENTS_OFFSET, NULL);
    if (v != Py_True) goto done;
    Py_DECREF(v);
    v = PyObject_VectorcallMethod(s_get_device, self, 1 | PY_VECTORCALL_ARGUMENTS_OFFSET, NULL);
    if (!v) goto done;
    *dev = PyLong_AsLong(v);
    if (*dev == -1 && PyErr_Occurred()) goto done;
    Py_DECREF(v);
    v = PyObject_VectorcallMethod(s_data_ptr, self, 1 | PY_VECTORCALL_ARGUMENTS_OFFSET, NULL);
    if (!v) goto done;
    *ptr = PyLong_AsVoidPtr(v);
    if (PyErr_Occurred()) goto done;
    ok = 1;
done:
    Py_XDECREF(v);
    Py_XDECREF(sh);
    if (!ok) PyErr_Clear();
    return ok;
}

/* The raw stream for `stream` (None: torch's current stream on dev; an
 * int: itself; else its cuda_stream attribute) in *out. Returns 0 when it
 * cannot be had (the error is cleared), 1 otherwise. */
static int stream_of(PyObject* stream, long dev, void** out) {
    PyObject* v;
    if (stream == Py_None) {
        PyObject* arg = PyLong_FromLong(dev);
        if (!arg) goto fail;
        PyObject* args[1] = {arg};
        v = PyObject_Vectorcall(g_raw_stream, args, 1, NULL);
        Py_DECREF(arg);
    } else if (PyLong_CheckExact(stream)) {
        Py_INCREF(stream);
        v = stream;
    } else {
        v = PyObject_GetAttr(stream, s_cuda_stream);
    }
    if (!v) goto fail;
    *out = PyLong_AsVoidPtr(v);
    Py_DECREF(v);
    if (PyErr_Occurred()) goto fail;
    return 1;
fail:
    PyErr_Clear();
    return 0;
}

static int current_device(long* dev) {
    PyObject* v = PyObject_Vectorcall(g_cur_device, NULL, 0, NULL);
    if (!v) {
        PyErr_Clear();
        return 0;
    }
    *dev = PyLong_AsLong(v);
    Py_DECREF(v);
    if (PyErr_Occurred()) {
        PyErr_Clear();
        return 0;
    }
    return 1;
}

/* Shared body: batch = 0 for score (q [D], C [K, D], out [K]), 1 for
 * score_batch (Q [B, D], C [B, K, D], out [B, K]). */
static PyObject* call(PyObject* const* args, Py_ssize_t nargs, int batch) {
    if (nargs != 8 || !g_single[0]) Py_RETURN_NONE;
    const int bc = PyObject_IsTrue(args[7]);
    if (bc < 0) {
        PyErr_Clear();
        Py_RETURN_NONE;
    }
    void *qp, *cp, *op, *st;
    long dq, dc, dout, cur;
    long long qs[3], cs[3], os[3];
    if (!facts(args[0], 1 + batch, 0, &qp, &dq, qs) || !facts(args[1], 2 + batch, bc, &cp, &dc, cs) ||
        !facts(args[2], 1 + batch, 0, &op, &dout, os))
        Py_RETURN_NONE;
    if (dq != dc || dout != dc || !current_device(&cur) || cur != dc) Py_RETURN_NONE;
    long long B = 1, K, D;
    if (batch) {
        B = cs[0];
        K = cs[1];
        D = cs[2];
        if (qs[0] != B || qs[1] != D || os[0] != B || os[1] != K) Py_RETURN_NONE;
    } else {
        K = cs[0];
        D = cs[1];
        if (qs[0] != D || os[0] != K) Py_RETURN_NONE;
    }
    if (B > INT32_MAX || K > INT32_MAX || D > INT32_MAX) Py_RETURN_NONE;
    const long normalize = PyLong_AsLong(args[3]);
    const double scale = PyFloat_AsDouble(args[4]), temperature = PyFloat_AsDouble(args[5]);
    if (PyErr_Occurred()) {
        PyErr_Clear();
        Py_RETURN_NONE;
    }
    if (normalize < INT32_MIN || normalize > INT32_MAX) Py_RETURN_NONE;
    if (!stream_of(args[6], dc, &st)) Py_RETURN_NONE;
    int s;
    if (batch)
        s = g_batch[bc](qp, cp, (int)B, (int)K, (int)D, (int)normalize, (float)scale, (float)temperature, op, st);
    else
        s = g_single[bc](qp, cp, (int)K, (int)D, (int)normalize, (float)scale, (float)temperature, op, st);
    return PyLong_FromLong(s);
}

static PyObject* py_score(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    return call(args, nargs, 0);
}

static PyObject* py_score_batch(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    return call(args, nargs, 1);
}

/* setup(single, batch, single_bf16, batch_bf16, float32, bfloat16,
 *       current_device, raw_stream): the library's entry points as
 *       addresses, the dtype objects and the two torch callables. */
static PyObject* py_setup(PyObject* self, PyObject* args) {
    (void)self;
    unsigned long long a[4];
    PyObject *f32, *bf16, *cur, *raw;
    if (!PyArg_ParseTuple(args, "KKKKOOOO", &a[0], &a[1], &a[2], &a[3], &f32, &bf16, &cur, &raw)) return NULL;
    if (!a[0] || !a[1] || !a[2] || !a[3] || !PyCallable_Check(cur) || !PyCallable_Check(raw)) {
        PyErr_SetString(PyExc_ValueError, "setup: null entry point or a non-callable");
        return NULL;
    }
    Py_XDECREF(g_f32);
    Py_XDECREF(g_bf16);
    Py_XDECREF(g_cur_device);
    Py_XDECREF(g_raw_stream);
    Py_INCREF(f32);
    Py_INCREF(bf16);
    Py_INCREF(cur);
    Py_INCREF(raw);
    g_f32 = f32;
    g_bf16 = bf16;
    g_cur_device = cur;
    g_raw_stream = raw;
    g_single[0] = (score1_fn)(uintptr_t)a[0];
    g_batch[0] = (scoreb_fn)(uintptr_t)a[1];
    g_single[1] = (score1_fn)(uintptr_t)a[2];
    g_batch[1] = (scoreb_fn)(uintptr_t)a[3];
    Py_RETURN_NONE;
}

static PyMethodDef methods[] = {
    {"setup", py_setup, METH_VARARGS, "Hand over the library's entry points and torch's objects."},
    {"score", (PyCFunction)(void (*)(void))py_score, METH_FASTCALL,
     "score(q, C, out, normalize, scale, temperature, stream, c_bf16) -> status, or None when not handled"},
    {"score_batch", (PyCFunction)(void (*)(void))py_score_batch, METH_FASTCALL,
     "score_batch(Q, C, out, normalize, scale, temperature, stream, c_bf16) -> status, or None when not handled"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_fastpath", NULL, -1, methods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastpath(void) {
    s_is_cuda = PyUnicode_InternFromString("is_cuda");
    s_dtype = PyUnicode_InternFromString("dtype");
    s_shape = PyUnicode_InternFromString("shape");
    s_is_contiguous = PyUnicode_InternFromString("is_contiguous");
    s_data_ptr = PyUnicode_InternFromString("data_ptr");
    s_get_device = PyUnicode_InternFromString("get_device");
    s_cuda_stream = PyUnicode_InternFromString("cuda_stream");
    if (!s_is_cuda || !s_dtype || !s_shape || !s_is_contiguous || !s_data_ptr || !s_get_device || !s_cuda_stream)
        return NULL;
    return PyModule_Create(&module);
}
