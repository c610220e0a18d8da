/* CPython fast path for the per-step calls of the Python binding:
 * pkd_plan, pkd_plan_shared and pkd_plan_cascade with the page tables passed as int32 arrays
 * through the buffer protocol, and pkd_run_scaled with its pointers as
 * integers (no per-argument ctypes conversion).  It only marshals arguments:
 * the entry points are the C ABI's own, whose addresses the binding hands
 * over once (init), so this module does not link libpkd.
 *
 * plan(ctx, indptr, indices, last, stream) -> (status, epoch)
 * plan_shared(ctx, group_indptr, indptr, indices, last, stream) -> (status, epoch)
 * plan_cascade(ctx, group_indptr, p_indptr, p_indices, p_last, s_indptr, s_indices, s_last,
 *              stream) -> (status, epoch)
 * run(ctx, q, kv, out, lse, k_scale, v_scale, expect_epoch, stream) -> status
 *
 * status is the C ABI's return value, or NOT_HANDLED (1000) when an argument
 * is not a 1-D C-contiguous int32 buffer: the caller then takes its general
 * path, which converts or rejects the input with a proper message. */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>
#include <string.h>

typedef int (*plan_fn)(void *ctx, const int32_t *indptr, const int32_t *indices,
                       const int32_t *last, int32_t batch, void *stream, uint64_t *epoch);
typedef int (*plan_shared_fn)(void *ctx, const int32_t *group_indptr, int32_t num_groups,
                              const int32_t *indptr, const int32_t *indices,
                              const int32_t *last, void *stream, uint64_t *epoch);

typedef int (*plan_cascade_fn)(void *ctx, const int32_t *group_indptr, int32_t num_groups,
                               const int32_t *p_indptr, const int32_t *p_indices,
                               const int32_t *p_last, const int32_t *s_indptr,
                               const int32_t *s_indices, const int32_t *s_last, void *stream,
                               uint64_t *epoch);

typedef int (*run_fn)(void *ctx, const void *q, const void *kv, void *out, float *lse,
                      float k_scale, float v_scale, uint64_t expect_epoch, void *stream);

static plan_fn g_plan = NULL;
static plan_shared_fn g_plan_shared = NULL;
static plan_cascade_fn g_plan_cascade = NULL;
static run_fn g_run = NULL;

#define NOT_HANDLED 1000
#define BAD_TABLE (-2)

static PyObject *init(PyObject *self, PyObject *args) {
  unsigned long long p, ps, pc = 0, pr = 0;
  (void)self;
  if (!PyArg_ParseTuple(args, "KK|KK", &p, &ps, &pc, &pr)) return NULL;
  g_plan = (plan_fn)(uintptr_t)p;
  g_plan_shared = (plan_shared_fn)(uintptr_t)ps;
  g_plan_cascade = (plan_cascade_fn)(uintptr_t)pc;
  g_run = (run_fn)(uintptr_t)pr;
  Py_RETURN_NONE;
}

/* The caller (the binding) has checked the tensors behind the pointers. */
static PyObject *run(PyObject *self, PyObject *args) {
  unsigned long long ctx, q, kv, out, lse, epoch, stream;
  float ks, vs;
  (void)self;
  if (!PyArg_ParseTuple(args, "KKKKKffKK", &ctx, &q, &kv, &out, &lse, &ks, &vs, &epoch, &stream))
    return NULL;
  if (g_run == NULL) return PyLong_FromLong(NOT_HANDLED);
  return PyLong_FromLong(g_run((void *)(uintptr_t)ctx, (const void *)(uintptr_t)q,
                               (const void *)(uintptr_t)kv, (void *)(uintptr_t)out,
                               (float *)(uintptr_t)lse, ks, vs, (uint64_t)epoch,
                               (void *)(uintptr_t)stream));
}

/* A 1-D C-contiguous buffer of 4-byte signed integers, or 0. */
static int get_i32(PyObject *obj, Py_buffer *view) {
  if (PyObject_GetBuffer(obj, view, PyBUF_C_CONTIGUOUS | PyBUF_FORMAT) != 0) {
    PyErr_Clear();
    return 0;
  }
  const char *f = view->format ? view->format : "B";
  if (f[0] == '<' || f[0] == '=' || f[0] == '@') ++f;
  if (view->ndim != 1 || view->itemsize != 4 || (strcmp(f, "i") != 0 && strcmp(f, "l") != 0)) {
    PyBuffer_Release(view);
    return 0;
  }
  return 1;
}

static PyObject *plan(PyObject *self, PyObject *args) {
  unsigned long long ctx, stream;
  PyObject *o_ip, *o_ix, *o_la;
  Py_buffer ip, ix, la;
  (void)self;
  if (!PyArg_ParseTuple(args, "KOOOK", &ctx, &o_ip, &o_ix, &o_la, &stream)) return NULL;
  if (g_plan == NULL) return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
  if (!get_i32(o_ip, &ip)) return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
  if (!get_i32(o_ix, &ix)) {
    PyBuffer_Release(&ip);
    return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
  }
  if (!get_i32(o_la, &la)) {
    PyBuffer_Release(&ip);
    PyBuffer_Release(&ix);
    return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
  }
  const Py_ssize_t batch = la.shape[0];
  int st;
  uint64_t epoch = 0;
  if (ip.shape[0] != batch + 1 || batch > INT32_MAX) {
    st = NOT_HANDLED;   /* the general path reports the shape error */
  } else if (batch > 0 && ix.shape[0] < ((const int32_t *)ip.buf)[batch]) {
    st = NOT_HANDLED;
  } else {
    st = g_plan((void *)(uintptr_t)ctx, (const int32_t *)ip.buf,
                ix.shape[0] ? (const int32_t *)ix.buf : NULL, (const int32_t *)la.buf,
                (int32_t)batch, (void *)(uintptr_t)stream, &epoch);
  }
  PyBuffer_Release(&ip);
  PyBuffer_Release(&ix);
  PyBuffer_Release(&la);
  return Py_BuildValue("iK", st, (unsigned long long)epoch);
}

static PyObject *plan_shared(PyObject *self, PyObject *args) {
  unsigned long long ctx, stream;
  PyObject *o_gi, *o_ip, *o_ix, *o_la;
  Py_buffer gi, ip, ix, la;
  (void)self;
  if (!PyArg_ParseTuple(args, "KOOOOK", &ctx, &o_gi, &o_ip, &o_ix, &o_la, &stream)) return NULL;
  if (g_plan_shared == NULL) return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
  PyObject *objs[4] = {o_gi, o_ip, o_ix, o_la};
  Py_buffer *views[4] = {&gi, &ip, &ix, &la};
  for (int k = 0; k < 4; ++k) {
    if (!get_i32(objs[k], views[k])) {
      for (int j = 0; j < k; ++j) PyBuffer_Release(views[j]);
      return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
    }
  }
  const Py_ssize_t groups = la.shape[0];
  int st;
  uint64_t epoch = 0;
  if (gi.shape[0] != groups + 1 || ip.shape[0] != groups + 1 || groups > INT32_MAX) {
    st = NOT_HANDLED;
  } else {
    st = g_plan_shared((void *)(uintptr_t)ctx, (const int32_t *)gi.buf, (int32_t)groups,
                       (const int32_t *)ip.buf, ix.shape[0] ? (const int32_t *)ix.buf : NULL,
                       (const int32_t *)la.buf, (void *)(uintptr_t)stream, &epoch);
  }
  for (int k = 0; k < 4; ++k) PyBuffer_Release(views[k]);
  return Py_BuildValue("iK", st, (unsigned long long)epoch);
}

static PyObject *plan_cascade(PyObject *self, PyObject *args) {
  unsigned long long ctx, stream;
  PyObject *objs[7];
  Py_buffer v[7];   /* group_indptr, prefix (indptr, indices, last), suffix (same) */
  (void)self;
  if (!PyArg_ParseTuple(args, "KOOOOOOOK", &ctx, &objs[0], &objs[1], &objs[2], &objs[3],
                        &objs[4], &objs[5], &objs[6], &stream))
    return NULL;
  if (g_plan_cascade == NULL) return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
  for (int k = 0; k < 7; ++k) {
    if (!get_i32(objs[k], &v[k])) {
      for (int j = 0; j < k; ++j) PyBuffer_Release(&v[j]);
      return Py_BuildValue("iK", NOT_HANDLED, 0ULL);
    }
  }
  const Py_ssize_t groups = v[3].shape[0], batch = v[6].shape[0];
  const int32_t *gi = (const int32_t *)v[0].buf;
  int st;
  uint64_t epoch = 0;
  if (v[0].shape[0] != groups + 1 || v[1].shape[0] != groups + 1 || v[4].shape[0] != batch + 1 ||
      groups > INT32_MAX || (groups > 0 && gi[groups] != batch) ||
      (groups > 0 && v[2].shape[0] < ((const int32_t *)v[1].buf)[groups]) ||
      (batch > 0 && v[5].shape[0] < ((const int32_t *)v[4].buf)[batch])) {
    st = NOT_HANDLED;
  } else {
    st = g_plan_cascade((void *)(uintptr_t)ctx, gi, (int32_t)groups, (const int32_t *)v[1].buf,
                        v[2].shape[0] ? (const int32_t *)v[2].buf : NULL,
                        (const int32_t *)v[3].buf, (const int32_t *)v[4].buf,
                        v[5].shape[0] ? (const int32_t *)v[5].buf : NULL,
                        (const int32_t *)v[6].buf, (void *)(uintptr_t)stream, &epoch);
  }
  for (int k = 0; k < 7; ++k) PyBuffer_Release(&v[k]);
  return Py_BuildValue("iK", st, (unsigned long long)epoch);
}

static PyMethodDef methods[] = {
    {"plan_cascade", plan_cascade, METH_VARARGS,
     "plan_cascade(ctx, group_indptr, p_indptr, p_indices, p_last, s_indptr, s_indices, "
     "s_last, stream) -> (status, epoch)"},
    {"init", init, METH_VARARGS,
     "init(plan_address, plan_shared_address[, plan_cascade_address[, run_scaled_address]])"},
    {"run", run, METH_VARARGS,
     "run(ctx, q, kv, out, lse, k_scale, v_scale, expect_epoch, stream) -> status"},
    {"plan", plan, METH_VARARGS, "plan(ctx, indptr, indices, last, stream) -> (status, epoch)"},
    {"plan_shared", plan_shared, METH_VARARGS,
     "plan_shared(ctx, group_indptr, indptr, indices, last, stream) -> (status, epoch)"},
    {NULL, NULL, 0, NULL}};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_pkd_plan", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__pkd_plan(void) { return PyModule_Create(&module); }
