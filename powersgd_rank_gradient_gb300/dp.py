"""Data-parallel PowerSGD across processes: one replica per process.

"DDP Communication Hooks", "PowerSGD Hooks", powerSGD_hook: every worker
computes its own P = M_w Q and Q = M_w^T P, and the hook allreduces the
uncompressed batch (step 2), the Ps (step 3.3) and the Qs (step 3.6);
"Default Communication Hooks", allreduce_hook: the allreduce is a mean.

``DataParallelPowerSGDState`` is one process's share of the job
(``psgd_dp_create``: this process's error-feedback residual and the shared
factors).  ``dp_powerSGD_hook`` runs one hook call: the library's three stages
(``psgd_dp_begin``, ``psgd_dp_project``, ``psgd_dp_finish``) with the process
group's SUM all-reduce of the two exchange buffers between them; the
library's kernels turn the sums into means and agree on a skipped step.  With
the NCCL backend the device buffers are reduced in place; with another
backend (gloo) through a host copy.  Every step of the method runs in the
library's CUDA kernels; this module only sequences them and the collectives.
"""

from __future__ import annotations

import ctypes

import torch
import torch.distributed as dist

from . import _lib
from ._lib import PSGD_BF16, PSGD_F16, PSGD_F32, check
from .hook import PowerSGDState, _numel, _stream_ptr


class _DeviceBuffer:
    """A device buffer of float32 owned by the library, seen by torch through
    the CUDA array interface (no copy)."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (int(n),), "typestr": "<f4", "data": (int(ptr), False),
                                         "version": 2}


class DataParallelPowerSGDState(PowerSGDState):
    """One process's share of a ``world_size``-process PowerSGD job.

    Keyword names and defaults are those of ``PowerSGDState`` ("PowerSGD
    State"); ``process_group`` (default: the default group) gives the world
    size and is the group ``dp_powerSGD_hook`` reduces over.  Introspection
    (``get_error(0)``, ``get_q``, ``get_p``, ``tensor_info``, ``stats``,
    ``status``) works as on ``PowerSGDState``.
    """

    def __init__(self, shapes, process_group=None, matrix_approximation_rank=1, start_powerSGD_iter=1000,
                 min_compression_rate=2, use_error_feedback=True, warm_start=True,
                 orthogonalization_epsilon=0.0, random_seed=0, batch_tensors_with_same_shape=False,
                 grad_dtype=torch.float32, device=None, world_size=None):
        if world_size is None:
            world_size = dist.get_world_size(process_group)
        if device is None:
            device = torch.cuda.current_device()
        device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        if grad_dtype not in (torch.float32, torch.float16, torch.bfloat16):
            raise ValueError("grad_dtype must be torch.float32, torch.float16 or torch.bfloat16")
        self.process_group = process_group
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        self.world_size = int(world_size)
        self.matrix_approximation_rank = int(matrix_approximation_rank)
        self.start_powerSGD_iter = int(start_powerSGD_iter)
        self.min_compression_rate = float(min_compression_rate)
        self.use_error_feedback = bool(use_error_feedback)
        self.warm_start = bool(warm_start)
        self.orthogonalization_epsilon = float(orthogonalization_epsilon)
        self.random_seed = int(random_seed)
        self.batch_tensors_with_same_shape = bool(batch_tensors_with_same_shape)
        self.grad_dtype = grad_dtype
        self.device = device
        self.numel = sum(_numel(s) for s in self.shapes)
        L = _lib.lib()
        d, n = _lib.shape_arrays(self.shapes)
        handle = ctypes.c_void_p()
        check(L.psgd_dp_create(
            d, n, len(self.shapes), self.world_size, self.matrix_approximation_rank,
            self.start_powerSGD_iter, self.min_compression_rate, int(self.use_error_feedback),
            int(self.warm_start), self.orthogonalization_epsilon, self.random_seed & (2**64 - 1),
            int(self.batch_tensors_with_same_shape),
            {torch.float16: PSGD_F16, torch.bfloat16: PSGD_BF16}.get(grad_dtype, PSGD_F32),
            device.index or 0, ctypes.byref(handle)))
        self._h = handle
        self._lib = L
        self._views = {}
        self._out = None
        self._grad = None

    def step(self, *args, **kwargs):
        raise RuntimeError("a data-parallel state steps through dp_powerSGD_hook (begin, project, finish)")

    def _view(self, ptr, n, out):
        if out is not None and ptr == out.data_ptr():
            return out[:n]
        key = (ptr, n)
        if key not in self._views:
            self._views[key] = torch.as_tensor(_DeviceBuffer(ptr, n), device=self.device)
        return self._views[key]

    # -- the three stages (torch's current stream) ------------------------------
    def begin(self, grad, out, inv_loss_scale=1.0):
        """psgd_dp_begin; returns the tensor to SUM-allreduce across the group."""
        if not (grad.is_cuda and grad.dtype == self.grad_dtype and grad.is_contiguous()
                and grad.numel() == self.numel):
            raise ValueError(f"grad must be a contiguous CUDA tensor of {self.numel} {self.grad_dtype} elements")
        if not (out.is_cuda and out.dtype == torch.float32 and out.is_contiguous() and out.numel() == self.numel):
            raise ValueError("out must be a contiguous CUDA float32 tensor of the bucket's size")
        ptr, cnt = ctypes.c_void_p(), ctypes.c_int64()
        check(self._lib.psgd_dp_begin(self._h, ctypes.c_void_p(grad.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                      float(inv_loss_scale), _stream_ptr(None), ctypes.byref(ptr),
                                      ctypes.byref(cnt)))
        self._out, self._grad = out, grad   # kept alive until finish
        if cnt.value == 0:
            return None
        return self._view(ptr.value, cnt.value, out)

    def project(self):
        """psgd_dp_project; returns the tensor to SUM-allreduce, or None."""
        ptr, cnt = ctypes.c_void_p(), ctypes.c_int64()
        check(self._lib.psgd_dp_project(self._h, _stream_ptr(None), ctypes.byref(ptr), ctypes.byref(cnt)))
        if cnt.value == 0:
            return None
        return self._view(ptr.value, cnt.value, None)

    def finish(self):
        """psgd_dp_finish: out holds the hook's result once the stream reaches it."""
        check(self._lib.psgd_dp_finish(self._h, _stream_ptr(None)))
        out = self._out
        self._out = self._grad = None
        return out


def allreduce_sum(t, group=None):
    """SUM-allreduce of ``t`` in place over ``group``: directly for NCCL or a
    host tensor, through a host copy for CUDA tensors on other backends."""
    if t is None or t.numel() == 0:
        return
    if not t.is_cuda or dist.get_backend(group) == "nccl":
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
        return
    h = t.cpu()
    dist.all_reduce(h, op=dist.ReduceOp.SUM, group=group)
    t.copy_(h)


def dp_powerSGD_hook(state, grad, out=None, inv_loss_scale=1.0, process_group=None):
    """One hook call ("PowerSGD Hooks", powerSGD_hook) on this process's
    replica bucket ``grad``; returns ``out``, the bucket every process
    receives.  ``state`` is a ``DataParallelPowerSGDState`` (or any object
    with its begin/project/finish stages); the exchanges are SUM all-reduces
    over ``process_group`` (default: the state's)."""
    group = process_group if process_group is not None else getattr(state, "process_group", None)
    if out is None:
        out = torch.empty(state.numel, dtype=torch.float32, device=grad.device)
    x = state.begin(grad, out, inv_loss_scale)
    allreduce_sum(x, group)
    y = state.project()
    allreduce_sum(y, group)
    state.finish()
    return out
