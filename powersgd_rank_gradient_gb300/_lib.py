"""ctypes binding of libpsgd.so (include/psgd.h): argument marshalling only.

Loading fails loudly when the library is missing; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpsgd.so")

PSGD_OK = 0
PSGD_SKIPPED_NONFINITE = 1
PSGD_EINVAL = -1
PSGD_ENOMEM = -2
PSGD_ECUDA = -3
PSGD_ETIMEOUT = -4
PSGD_F32 = 0
PSGD_F16 = 1
PSGD_BF16 = 2
PSGD_MAX_RANK = 32
PSGD_MAX_WORLD = 64
PSGD_MAX_GROUP_STREAMS = 16

# every symbol include/psgd.h declares
EXPORTS = [
    "psgd_plan", "psgd_state_create", "psgd_state_create_batched", "psgd_state_destroy",
    "psgd_step", "psgd_step_host",
    "psgd_step_status", "psgd_get_stats", "psgd_tensor_info", "psgd_error_numel", "psgd_set_q",
    "psgd_get_q", "psgd_get_p", "psgd_get_error", "psgd_set_error", "psgd_workspace_bytes",
    "psgd_set_error_store_halves", "psgd_profile", "psgd_profile_select", "psgd_profile_kinds", "psgd_profile_read", "psgd_last_error",
    "psgd_project_q_static",
    "psgd_group_create", "psgd_group_destroy", "psgd_group_step", "psgd_group_wait",
    "psgd_group_status", "psgd_group_bucket", "psgd_group_size", "psgd_set_graph", "psgd_graph_stats",
    "psgd_dp_create", "psgd_dp_begin", "psgd_dp_project", "psgd_dp_finish", "psgd_build_id",
]

_lib = None


class PsgdError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"psgd error {code}: {msg}")
        self.code = code


def lib():
    """The loaded library (loaded once).  Raises if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    c_i32, c_i64, c_u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    P = ctypes.c_void_p
    pi64 = ctypes.POINTER(c_i64)
    pi32 = ctypes.POINTER(c_i32)
    L.psgd_plan.argtypes = [pi64, pi32, c_i32, c_i32, ctypes.c_double, pi32, pi32, pi64, pi64]
    L.psgd_plan.restype = ctypes.c_int
    L.psgd_state_create.argtypes = [pi64, pi32, c_i32, c_i32, c_i32, c_i64, ctypes.c_double, c_i32,
                                    c_i32, ctypes.c_float, c_u64, c_i32, ctypes.c_int, c_i32,
                                    ctypes.POINTER(P)]
    L.psgd_state_create.restype = ctypes.c_int
    L.psgd_state_create_batched.argtypes = [c_i64, c_i32, c_i32, c_i64, c_i32, c_i32, ctypes.c_float,
                                            c_u64, ctypes.c_int, c_i32, ctypes.POINTER(P)]
    L.psgd_state_create_batched.restype = ctypes.c_int
    L.psgd_state_destroy.argtypes = [P]
    L.psgd_state_destroy.restype = None
    L.psgd_step.argtypes = [P, ctypes.POINTER(P), P, ctypes.c_float, P]
    L.psgd_step.restype = ctypes.c_int
    L.psgd_step_host.argtypes = [P, ctypes.POINTER(P), P, ctypes.c_float, P]
    L.psgd_step_host.restype = ctypes.c_int
    L.psgd_step_status.argtypes = [P, P]
    L.psgd_step_status.restype = ctypes.c_int
    L.psgd_get_stats.argtypes = [P, pi64, pi64, pi64]
    L.psgd_get_stats.restype = ctypes.c_int
    L.psgd_tensor_info.argtypes = [P, c_i32, pi32, pi64, pi64, pi32, pi64, pi64]
    L.psgd_tensor_info.restype = ctypes.c_int
    L.psgd_error_numel.argtypes = [P]
    L.psgd_error_numel.restype = c_i64
    L.psgd_set_q.argtypes = [P, c_i32, P, c_i32]
    L.psgd_set_q.restype = ctypes.c_int
    L.psgd_get_q.argtypes = [P, c_i32, P]
    L.psgd_get_q.restype = ctypes.c_int
    L.psgd_get_p.argtypes = [P, c_i32, P]
    L.psgd_get_p.restype = ctypes.c_int
    L.psgd_get_error.argtypes = [P, c_i32, P, P]
    L.psgd_get_error.restype = ctypes.c_int
    L.psgd_set_error.argtypes = [P, c_i32, P, P]
    L.psgd_set_error.restype = ctypes.c_int
    L.psgd_workspace_bytes.argtypes = [P]
    L.psgd_workspace_bytes.restype = ctypes.c_size_t
    L.psgd_profile.argtypes = [P, c_i32]
    L.psgd_profile.restype = ctypes.c_int
    L.psgd_set_error_store_halves.argtypes = [P, c_i32]
    L.psgd_set_error_store_halves.restype = ctypes.c_int
    L.psgd_profile_select.argtypes = [P, ctypes.c_uint32]
    L.psgd_profile_select.restype = ctypes.c_int
    L.psgd_profile_kinds.argtypes = []
    L.psgd_profile_kinds.restype = c_i32
    L.psgd_profile_read.argtypes = [P, c_i32, ctypes.POINTER(ctypes.c_char_p), pi64,
                                    ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    L.psgd_profile_read.restype = ctypes.c_int
    L.psgd_project_q_static.argtypes = [P, P, P, c_i64, c_i64, c_i32, P]
    L.psgd_project_q_static.restype = ctypes.c_int
    L.psgd_group_create.argtypes = [c_i32, pi32, pi64, pi32, c_i32, c_i32, c_i64, ctypes.c_double, c_i32,
                                    c_i32, ctypes.c_float, c_u64, c_i32, ctypes.c_int, c_i32, c_i32,
                                    ctypes.POINTER(P)]
    L.psgd_group_create.restype = ctypes.c_int
    L.psgd_group_destroy.argtypes = [P]
    L.psgd_group_destroy.restype = None
    L.psgd_group_step.argtypes = [P, c_i32, ctypes.POINTER(P), P, ctypes.c_float, P]
    L.psgd_group_step.restype = ctypes.c_int
    L.psgd_group_wait.argtypes = [P, P]
    L.psgd_group_wait.restype = ctypes.c_int
    L.psgd_group_status.argtypes = [P, P]
    L.psgd_group_status.restype = ctypes.c_int
    L.psgd_group_bucket.argtypes = [P, c_i32, ctypes.POINTER(P)]
    L.psgd_group_bucket.restype = ctypes.c_int
    L.psgd_group_size.argtypes = [P]
    L.psgd_group_size.restype = c_i32
    L.psgd_set_graph.argtypes = [P, c_i32]
    L.psgd_set_graph.restype = ctypes.c_int
    L.psgd_graph_stats.argtypes = [P, pi64, pi64]
    L.psgd_graph_stats.restype = ctypes.c_int
    L.psgd_dp_create.argtypes = L.psgd_state_create.argtypes
    L.psgd_dp_create.restype = ctypes.c_int
    pf = ctypes.POINTER(ctypes.c_void_p)
    L.psgd_dp_begin.argtypes = [P, P, P, ctypes.c_float, P, pf, pi64]
    L.psgd_dp_begin.restype = ctypes.c_int
    L.psgd_dp_project.argtypes = [P, P, pf, pi64]
    L.psgd_dp_project.restype = ctypes.c_int
    L.psgd_dp_finish.argtypes = [P, P]
    L.psgd_dp_finish.restype = ctypes.c_int
    L.psgd_build_id.argtypes = []
    L.psgd_build_id.restype = ctypes.c_char_p
    L.psgd_last_error.argtypes = []
    L.psgd_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def check(rc):
    """Raise PsgdError for a negative return code; pass others through."""
    if rc < 0:
        raise PsgdError(rc, lib().psgd_last_error().decode())
    return rc


def shape_arrays(shapes):
    dims = [int(d) for s in shapes for d in s]
    ndims = [len(s) for s in shapes]
    d = (ctypes.c_int64 * max(1, len(dims)))(*dims)
    n = (ctypes.c_int32 * max(1, len(ndims)))(*ndims)
    return d, n


def plan(shapes, matrix_approximation_rank, min_compression_rate):
    """psgd_plan: host-only gate.  Returns (compressed, ranks, rows, cols) lists."""
    L = lib()
    d, n = shape_arrays(shapes)
    k = max(1, len(shapes))
    comp = (ctypes.c_int32 * k)()
    ranks = (ctypes.c_int32 * k)()
    rows = (ctypes.c_int64 * k)()
    cols = (ctypes.c_int64 * k)()
    check(L.psgd_plan(d, n, len(shapes), int(matrix_approximation_rank), float(min_compression_rate),
                      comp, ranks, rows, cols))
    m = len(shapes)
    return list(comp)[:m], list(ranks)[:m], list(rows)[:m], list(cols)[:m]
