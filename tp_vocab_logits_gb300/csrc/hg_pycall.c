/*
 * _hgcall: a CPython object that holds the marshalled arguments of one
 * hg_gather call (handle, shard and output pointer arrays, row count, stream)
 * and makes the call when invoked.
 *
 * It exists for the host cost per call only. Through ctypes, every call
 * converts five arguments and costs about 1 us of interpreter time on top of
 * the C entry point; a decode loop that issues one gather per step pays that
 * on every step. This object calls the entry point directly from tp_call.
 *
 * It computes nothing: the pointers come from the Python binding, which has
 * already checked the tensors, and the C entry point validates them again.
 * The entry point's address is passed in by the binding (from the loaded
 * libhg), so this module does not link against libhg itself.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include <stdint.h>
#include <stdlib.h>

typedef int (*gather_fn)(void *h, const void *const *shards, void *const *outs, int M,
                         void *stream);

typedef struct {
  PyObject_HEAD
  gather_fn fn;
  PyObject *handle;   /* the binding's Handle: its `ptr` attribute is read at each call */
  const void **shards;
  void **outs;
  int M;
  void *stream;
  PyObject *keep;     /* keeps the tensors behind the pointers alive */
  PyObject *on_error; /* called with the status when the call fails; raises */
} CallObject;

static PyObject *g_ptr_name; /* interned "ptr" */

static int read_ptrs(PyObject *seq, void ***out, Py_ssize_t *n) {
  PyObject *fast = PySequence_Fast(seq, "pointer list must be a sequence of ints");
  if (!fast) return -1;
  *n = PySequence_Fast_GET_SIZE(fast);
  *out = (void **)calloc((size_t)(*n > 0 ? *n : 1), sizeof(void *));
  if (!*out) {
    Py_DECREF(fast);
    PyErr_NoMemory();
    return -1;
  }
  for (Py_ssize_t i = 0; i < *n; ++i) {
    void *p = PyLong_AsVoidPtr(PySequence_Fast_GET_ITEM(fast, i));
    if (!p && PyErr_Occurred()) {
      Py_DECREF(fast);
      return -1;
    }
    (*out)[i] = p;
  }
  Py_DECREF(fast);
  return 0;
}

static void call_dealloc(CallObject *self) {
  free((void *)self->shards);
  free(self->outs);
  Py_XDECREF(self->handle);
  Py_XDECREF(self->keep);
  Py_XDECREF(self->on_error);
  Py_TYPE(self)->tp_free((PyObject *)self);
}

/* Call(fn_address, handle, shard_ptrs, out_ptrs, M, stream, keep, on_error) */
static PyObject *call_new(PyTypeObject *type, PyObject *args, PyObject *kwds) {
  PyObject *fn_obj, *handle, *shard_seq, *out_seq, *stream_obj, *keep, *on_error;
  int M;
  if (kwds && PyDict_Size(kwds) > 0) {
    PyErr_SetString(PyExc_TypeError, "Call takes positional arguments only");
    return NULL;
  }
  if (!PyArg_ParseTuple(args, "OOOOiOOO", &fn_obj, &handle, &shard_seq, &out_seq, &M,
                        &stream_obj, &keep, &on_error))
    return NULL;
  if (!PyCallable_Check(on_error)) {
    PyErr_SetString(PyExc_TypeError, "on_error must be callable");
    return NULL;
  }
  void *fn = PyLong_AsVoidPtr(fn_obj);
  if (!fn) {
    if (!PyErr_Occurred()) PyErr_SetString(PyExc_ValueError, "null function address");
    return NULL;
  }
  void *stream = PyLong_AsVoidPtr(stream_obj);
  if (!stream && PyErr_Occurred()) return NULL;
  CallObject *self = (CallObject *)type->tp_alloc(type, 0);
  if (!self) return NULL;
  Py_ssize_t ns = 0, no = 0;
  void **shards = NULL;
  if (read_ptrs(shard_seq, &shards, &ns) != 0 || read_ptrs(out_seq, &self->outs, &no) != 0) {
    free(shards);
    Py_DECREF(self);
    return NULL;
  }
  self->shards = (const void **)shards;
  if (ns != no) {
    Py_DECREF(self);
    PyErr_SetString(PyExc_ValueError, "shard and output lists differ in length");
    return NULL;
  }
  self->fn = (gather_fn)fn;
  self->M = M;
  self->stream = stream;
  Py_INCREF(handle);
  self->handle = handle;
  Py_INCREF(keep);
  self->keep = keep;
  Py_INCREF(on_error);
  self->on_error = on_error;
  return (PyObject *)self;
}

static PyObject *call_call(PyObject *obj, PyObject *args, PyObject *kwds) {
  CallObject *self = (CallObject *)obj;
  if ((args && PyTuple_GET_SIZE(args) != 0) || (kwds && PyDict_Size(kwds) != 0)) {
    PyErr_SetString(PyExc_TypeError, "a gather call takes no arguments");
    return NULL;
  }
  /* A closed handle has ptr 0 (None is taken the same way): pass NULL, which
     the library rejects. */
  PyObject *p = PyObject_GetAttr(self->handle, g_ptr_name);
  if (!p) return NULL;
  void *h = p == Py_None ? NULL : PyLong_AsVoidPtr(p);
  Py_DECREF(p);
  if (!h && PyErr_Occurred()) return NULL;
  const int st = self->fn(h, self->shards, (void *const *)self->outs, self->M, self->stream);
  if (st != 0) {
    PyObject *r = PyObject_CallFunction(self->on_error, "i", st);
    if (!r) return NULL;
    Py_DECREF(r);
    PyErr_Format(PyExc_RuntimeError, "hg_gather failed with status %d", st);
    return NULL;
  }
  Py_RETURN_NONE;
}

static PyTypeObject CallType = {
    PyVarObject_HEAD_INIT(NULL, 0)
    .tp_name = "_hgcall.Call",
    .tp_basicsize = sizeof(CallObject),
    .tp_dealloc = (destructor)call_dealloc,
    .tp_call = call_call,
    .tp_flags = Py_TPFLAGS_DEFAULT,
    .tp_doc = "Marshalled arguments of one hg_gather call; calling it makes the call.",
    .tp_new = call_new,
};

static struct PyModuleDef hgcall_module = {
    PyModuleDef_HEAD_INIT, "_hgcall", "Direct hg_gather calls for the Python binding.", -1,
    NULL /* methods */, NULL /* slots */, NULL /* traverse */, NULL /* clear */, NULL /* free */,
};

PyMODINIT_FUNC PyInit__hgcall(void) {
  if (PyType_Ready(&CallType) < 0) return NULL;
  g_ptr_name = PyUnicode_InternFromString("ptr");
  if (!g_ptr_name) return NULL;
  PyObject *m = PyModule_Create(&hgcall_module);
  if (!m) return NULL;
  Py_INCREF(&CallType);
  if (PyModule_AddObject(m, "Call", (PyObject *)&CallType) < 0) {
    Py_DECREF(&CallType);
    Py_DECREF(m);
    return NULL;
  }
  return m;
}
