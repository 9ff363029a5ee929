"""Python face of the library: ``PowerSGDState`` and ``powerSGD_hook``.

Names and defaults follow "DDP Communication Hooks" (PyTorch 1.11 docs),
"PowerSGD State": ``PowerSGDState(process_group, matrix_approximation_rank=1,
start_powerSGD_iter=1000, min_compression_rate=2, use_error_feedback=True,
warm_start=True, orthogonalization_epsilon=0, random_seed=0, ...)`` plus
``batch_tensors_with_same_shape`` from the later page.  The process group is
replaced by ``world_size`` simulated replicas on one GPU.  torch is used only
for device memory and streams; every step of the method runs in the CUDA
kernels of libpsgd.so.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import PSGD_BF16, PSGD_F16, PSGD_F32, PSGD_SKIPPED_NONFINITE, check


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class PowerSGDState:
    """Hyper-parameters and device state of the hook for one bucket layout."""

    def __init__(self, shapes, world_size, matrix_approximation_rank=1, start_powerSGD_iter=1000,
                 min_compression_rate=2, use_error_feedback=True, warm_start=True,
                 orthogonalization_epsilon=0.0, random_seed=0, batch_tensors_with_same_shape=False,
                 grad_dtype=torch.float32, device=None):
        if device is None:
            device = torch.cuda.current_device()
        device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        if grad_dtype not in (torch.float32, torch.float16, torch.bfloat16):
            raise ValueError("grad_dtype must be torch.float32, torch.float16 or torch.bfloat16")
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
        check(L.psgd_state_create(
            d, n, len(self.shapes), self.world_size, self.matrix_approximation_rank,
            self.start_powerSGD_iter, self.min_compression_rate, int(self.use_error_feedback),
            int(self.warm_start), self.orthogonalization_epsilon, self.random_seed & (2**64 - 1),
            int(self.batch_tensors_with_same_shape),
            {torch.float16: PSGD_F16, torch.bfloat16: PSGD_BF16}.get(grad_dtype, PSGD_F32),
            device.index or 0,
            ctypes.byref(handle)))
        self._h = handle
        self._lib = L

    # -- lifetime -------------------------------------------------------------
    def close(self):
        if getattr(self, "_owner", None) is not None:
            self._h = ctypes.c_void_p()   # a group's bucket: the group frees it
            return
        if getattr(self, "_h", None) and self._h.value:
            self._lib.psgd_state_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- the hook -------------------------------------------------------------
    def step(self, grads, out=None, inv_loss_scale=1.0, stream=None):
        """Enqueue one hook call on the W replica buckets; returns ``out``."""
        if len(grads) != self.world_size:
            raise ValueError(f"expected {self.world_size} replica buckets, got {len(grads)}")
        for g in grads:
            if not (g.is_cuda and g.dtype == self.grad_dtype and g.is_contiguous() and g.numel() == self.numel):
                raise ValueError("each replica bucket must be a contiguous CUDA tensor of "
                                 f"{self.numel} {self.grad_dtype} elements")
        if out is None:
            out = torch.empty(self.numel, dtype=torch.float32, device=self.device)
        if not (out.is_cuda and out.dtype == torch.float32 and out.is_contiguous() and out.numel() == self.numel):
            raise ValueError("out must be a contiguous CUDA float32 tensor of the bucket's size")
        ptrs = (ctypes.c_void_p * self.world_size)(*[g.data_ptr() for g in grads])
        check(self._lib.psgd_step(self._h, ptrs, ctypes.c_void_p(out.data_ptr()), float(inv_loss_scale),
                                  _stream_ptr(stream)))
        return out

    def step_host(self, host_grads, host_out, inv_loss_scale=1.0, stream=None):
        """psgd_step_host: host (ideally pinned) CPU tensors in and out."""
        ptrs = (ctypes.c_void_p * self.world_size)(*[g.data_ptr() for g in host_grads])
        check(self._lib.psgd_step_host(self._h, ptrs, ctypes.c_void_p(host_out.data_ptr()),
                                       float(inv_loss_scale), _stream_ptr(stream)))
        return host_out

    def status(self, stream=None):
        """Synchronises and returns True when the last step was skipped (inf/NaN)."""
        rc = check(self._lib.psgd_step_status(self._h, _stream_ptr(stream)))
        return rc == PSGD_SKIPPED_NONFINITE

    def set_graph(self, enable=True):
        """psgd_set_graph: replay the steady compressed step as a CUDA graph."""
        check(self._lib.psgd_set_graph(self._h, int(bool(enable))))

    def graph_stats(self):
        """(captures, replays) of the steady-step graph."""
        c, r = ctypes.c_int64(), ctypes.c_int64()
        check(self._lib.psgd_graph_stats(self._h, ctypes.byref(c), ctypes.byref(r)))
        return c.value, r.value

    # -- introspection ----------------------------------------------------------
    def stats(self):
        b, a, it = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check(self._lib.psgd_get_stats(self._h, ctypes.byref(b), ctypes.byref(a), ctypes.byref(it)))
        return b.value, a.value, it.value

    def tensor_info(self, t):
        c, r, k = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64()
        rows, cols, boff, poff = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check(self._lib.psgd_tensor_info(self._h, int(t), ctypes.byref(c), ctypes.byref(rows),
                                         ctypes.byref(cols), ctypes.byref(r), ctypes.byref(boff),
                                         ctypes.byref(poff)))
        return dict(compressed=bool(c.value), rows=rows.value, cols=cols.value, rank=r.value,
                    bucket_offset=boff.value, packed_offset=poff.value)

    def error_numel(self):
        return int(self._lib.psgd_error_numel(self._h))

    def workspace_bytes(self):
        return int(self._lib.psgd_workspace_bytes(self._h))

    def set_error_store_halves(self, halves):
        """psgd_set_error_store_halves: 1 keeps the error-feedback store once
        (the pages' memory; a skipped inf/NaN step then leaves the error
        feedback changed), 2 (default) twice.  Before the first step."""
        check(self._lib.psgd_set_error_store_halves(self._h, int(halves)))

    def set_q(self, t, q, is_draw=True):
        q = torch.as_tensor(q, dtype=torch.float32).contiguous().cpu()
        check(self._lib.psgd_set_q(self._h, int(t), ctypes.c_void_p(q.data_ptr()), int(is_draw)))

    def get_q(self, t):
        info = self.tensor_info(t)
        out = torch.empty(info["cols"], info["rank"], dtype=torch.float32)
        check(self._lib.psgd_get_q(self._h, int(t), ctypes.c_void_p(out.data_ptr())))
        return out

    def get_p(self, t):
        info = self.tensor_info(t)
        out = torch.empty(info["rows"], info["rank"], dtype=torch.float32)
        check(self._lib.psgd_get_p(self._h, int(t), ctypes.c_void_p(out.data_ptr())))
        return out

    def get_error(self, replica, out=None, stream=None):
        n = self.error_numel()
        if out is None:
            out = torch.empty(max(1, n), dtype=torch.float32, device=self.device)
        check(self._lib.psgd_get_error(self._h, int(replica), ctypes.c_void_p(out.data_ptr()),
                                       _stream_ptr(stream)))
        return out[:n]

    def set_error(self, replica, e, stream=None):
        e = e.to(device=self.device, dtype=torch.float32).contiguous()
        check(self._lib.psgd_set_error(self._h, int(replica), ctypes.c_void_p(e.data_ptr()),
                                       _stream_ptr(stream)))

    # -- measurement ------------------------------------------------------------
    def profile(self, enable=True):
        check(self._lib.psgd_profile(self._h, int(enable)))

    def profile_select(self, kinds):
        """psgd_profile_select: record only the named kernel kinds (an empty
        list stops recording)."""
        names = self.profile_kind_names()
        mask = 0
        for k in kinds:
            mask |= 1 << names.index(k)
        check(self._lib.psgd_profile_select(self._h, mask))

    def profile_kind_names(self):
        """The kernel kinds' names, in kind order."""
        names = []
        for k in range(self._lib.psgd_profile_kinds()):
            name = ctypes.c_char_p()
            # no launches / time pointers: the name only, the record stays
            check(self._lib.psgd_profile_read(self._h, k, ctypes.byref(name), None, None, None))
            names.append(name.value.decode())
        return names

    def profile_read(self):
        """{kind: (launches, total_ms, algorithmic bytes per launch)} since the last read."""
        res = {}
        for k in range(self._lib.psgd_profile_kinds()):
            name = ctypes.c_char_p()
            n = ctypes.c_int64()
            ms = ctypes.c_double()
            by = ctypes.c_double()
            check(self._lib.psgd_profile_read(self._h, k, ctypes.byref(name), ctypes.byref(n),
                                              ctypes.byref(ms), ctypes.byref(by)))
            res[name.value.decode()] = (n.value, ms.value, by.value)
        return res


class BatchedPowerSGDState(PowerSGDState):
    """State of batched_powerSGD_hook ("PowerSGD Hooks"): the whole flat
    bucket of ``numel`` elements is compressed as one zero-padded square
    matrix of side ceil(sqrt(numel)); the result is truncated to ``numel``."""

    def __init__(self, numel, world_size, matrix_approximation_rank=1, start_powerSGD_iter=1000,
                 use_error_feedback=True, warm_start=True, orthogonalization_epsilon=0.0,
                 random_seed=0, grad_dtype=torch.float32, device=None):
        if device is None:
            device = torch.cuda.current_device()
        device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        if grad_dtype not in (torch.float32, torch.float16, torch.bfloat16):
            raise ValueError("grad_dtype must be torch.float32, torch.float16 or torch.bfloat16")
        self.shapes = None
        self.world_size = int(world_size)
        self.matrix_approximation_rank = int(matrix_approximation_rank)
        self.start_powerSGD_iter = int(start_powerSGD_iter)
        self.min_compression_rate = 0.0
        self.use_error_feedback = bool(use_error_feedback)
        self.warm_start = bool(warm_start)
        self.orthogonalization_epsilon = float(orthogonalization_epsilon)
        self.random_seed = int(random_seed)
        self.batch_tensors_with_same_shape = False
        self.grad_dtype = grad_dtype
        self.device = device
        self.numel = int(numel)
        L = _lib.lib()
        handle = ctypes.c_void_p()
        check(L.psgd_state_create_batched(
            self.numel, self.world_size, self.matrix_approximation_rank, self.start_powerSGD_iter,
            int(self.use_error_feedback), int(self.warm_start), self.orthogonalization_epsilon,
            self.random_seed & (2**64 - 1),
            {torch.float16: PSGD_F16, torch.bfloat16: PSGD_BF16}.get(grad_dtype, PSGD_F32),
            device.index or 0, ctypes.byref(handle)))
        self._h = handle
        self._lib = L
        self.side = self.tensor_info(0)["rows"]


class PowerSGDGroup:
    """Per-bucket PowerSGD states stepped on several CUDA streams ("DDP
    Communication Hooks", "What Does a Communication Hook Operate On?": the
    hook runs once per gradient bucket, and bucketing lets one bucket's work
    overlap another's).  ``bucket_shapes[b]`` lists bucket b's tensor shapes;
    the keyword arguments are PowerSGDState's and apply to every bucket.
    ``graphs``: replay each bucket's steady step as a CUDA graph (the buckets'
    buffers must then stay the same from step to step to avoid recaptures)."""

    def __init__(self, bucket_shapes, world_size, matrix_approximation_rank=1, start_powerSGD_iter=1000,
                 min_compression_rate=2, use_error_feedback=True, warm_start=True,
                 orthogonalization_epsilon=0.0, random_seed=0, batch_tensors_with_same_shape=False,
                 grad_dtype=torch.float32, n_streams=8, graphs=True, device=None):
        if device is None:
            device = torch.cuda.current_device()
        device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        if grad_dtype not in (torch.float32, torch.float16, torch.bfloat16):
            raise ValueError("grad_dtype must be torch.float32, torch.float16 or torch.bfloat16")
        self.bucket_shapes = [[tuple(int(d) for d in sh) for sh in b] for b in bucket_shapes]
        self.world_size = int(world_size)
        self.grad_dtype = grad_dtype
        self.device = device
        self.n_streams = int(n_streams)
        L = _lib.lib()
        flat = [sh for b in self.bucket_shapes for sh in b]
        d, n = _lib.shape_arrays(flat)
        counts = (ctypes.c_int32 * max(1, len(self.bucket_shapes)))(*[len(b) for b in self.bucket_shapes])
        handle = ctypes.c_void_p()
        check(L.psgd_group_create(
            len(self.bucket_shapes), counts, d, n, self.world_size, int(matrix_approximation_rank),
            int(start_powerSGD_iter), float(min_compression_rate), int(bool(use_error_feedback)),
            int(bool(warm_start)), float(orthogonalization_epsilon), int(random_seed) & (2**64 - 1),
            int(bool(batch_tensors_with_same_shape)),
            {torch.float16: PSGD_F16, torch.bfloat16: PSGD_BF16}.get(grad_dtype, PSGD_F32),
            self.n_streams, device.index or 0, ctypes.byref(handle)))
        self._h = handle
        self._lib = L
        self.buckets = [self._bucket_view(b) for b in range(len(self.bucket_shapes))]
        # the steady step of every bucket as one CUDA graph launch (psgd_set_graph)
        for v in self.buckets:
            v.set_graph(graphs)

    def _bucket_view(self, b):
        h = ctypes.c_void_p()
        check(self._lib.psgd_group_bucket(self._h, b, ctypes.byref(h)))
        v = PowerSGDState.__new__(PowerSGDState)
        v._h, v._lib, v._owner = h, self._lib, self
        v.shapes = self.bucket_shapes[b]
        v.world_size = self.world_size
        v.grad_dtype = self.grad_dtype
        v.device = self.device
        v.numel = sum(_numel(sh) for sh in v.shapes)
        return v

    def __len__(self):
        return len(self.bucket_shapes)

    def step(self, bucket, grads, out=None, inv_loss_scale=1.0, stream=None):
        """Enqueue bucket ``bucket``'s hook call; returns ``out`` (valid after wait())."""
        v = self.buckets[bucket]
        if len(grads) != self.world_size:
            raise ValueError(f"expected {self.world_size} replica buckets, got {len(grads)}")
        for g in grads:
            if not (g.is_cuda and g.dtype == self.grad_dtype and g.is_contiguous() and g.numel() == v.numel):
                raise ValueError(f"bucket {bucket}: each replica bucket must be a contiguous CUDA tensor of "
                                 f"{v.numel} {self.grad_dtype} elements")
        if out is None:
            out = torch.empty(v.numel, dtype=torch.float32, device=self.device)
        if not (out.is_cuda and out.dtype == torch.float32 and out.is_contiguous() and out.numel() == v.numel):
            raise ValueError("out must be a contiguous CUDA float32 tensor of the bucket's size")
        ptrs = (ctypes.c_void_p * self.world_size)(*[g.data_ptr() for g in grads])
        check(self._lib.psgd_group_step(self._h, int(bucket), ptrs, ctypes.c_void_p(out.data_ptr()),
                                        float(inv_loss_scale), _stream_ptr(stream)))
        return out

    def wait(self, stream=None):
        """Make ``stream`` (default: the current stream) wait for every enqueued bucket step."""
        check(self._lib.psgd_group_wait(self._h, _stream_ptr(stream)))

    def status(self, stream=None):
        """Synchronises; True when any bucket's last step was skipped (inf/NaN)."""
        return check(self._lib.psgd_group_status(self._h, _stream_ptr(stream))) == PSGD_SKIPPED_NONFINITE

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            for v in getattr(self, "buckets", []):
                v._h = ctypes.c_void_p()
            self._lib.psgd_group_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def batched_powerSGD_hook(state, grads, out=None, inv_loss_scale=1.0, stream=None):
    """One call of batched_powerSGD_hook ("PowerSGD Hooks") on the W replica buckets."""
    return state.step(grads, out=out, inv_loss_scale=inv_loss_scale, stream=stream)


def powerSGD_hook(state, grads, out=None, inv_loss_scale=1.0, stream=None):
    """One hook call ("PowerSGD Hooks", powerSGD_hook) on the W replica buckets."""
    return state.step(grads, out=out, inv_loss_scale=inv_loss_scale, stream=stream)


def _numel(shape):
    n = 1
    for d in shape:
        n *= int(d)
    return n
