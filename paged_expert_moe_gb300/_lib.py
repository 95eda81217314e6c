"""ctypes binding of libpagedmoe.so (include/pagedmoe.h): argument marshalling only.

Every function keeps the C name. Tensors are passed as raw device pointers
(``tensor.data_ptr()``) with the current torch CUDA stream; every step of the
layer runs in the library's own CUDA kernels. If the library is missing, loading
fails with an error (there is no fallback path).
"""

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedmoe.so")

PMOE_OK, PMOE_EINVAL, PMOE_ENOMEM, PMOE_EHOSTALLOC, PMOE_ECUDA, PMOE_EUNSUPPORTED, PMOE_ETIMEOUT, PMOE_EDEVICE = \
    0, -1, -2, -3, -4, -5, -6, -7
PMOE_BF16, PMOE_FP8_BLOCK128, PMOE_INT4_GPTQ_G128, PMOE_MXFP4, PMOE_NVFP4 = 0, 1, 2, 3, 4
PMOE_PAGEIN_COPY_ENGINE, PMOE_PAGEIN_SM_PULL = 0, 1


class PmoeError(RuntimeError):
    def __init__(self, status, what):
        lib = _LIB
        text = lib.pmoe_status_string(status).decode() if lib else str(status)
        detail = lib.pmoe_last_error().decode() if lib else ""
        super().__init__(f"{what}: {text} ({status}) {detail}".strip())
        self.status = status


class pmoe_cache_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_experts", "top_k", "hidden", "intermediate", "num_slots", "num_layers", "format",
        "max_tokens", "pagein_mode", "device")]


class pmoe_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("steps", "hits", "misses", "waves", "bytes_paged")]


class pmoe_kernel_times(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * 12), ("launches", ctypes.c_uint64 * 12), ("copies", ctypes.c_uint64)]


KERNEL_CLASSES = ("residency", "group", "gather", "gateup", "down", "combine", "pull", "pagein_copy", "decode")

_LIB = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "pmoe_version": ([], _I),
    "pmoe_status_string": ([_I], ctypes.c_char_p),
    "pmoe_last_error": ([], ctypes.c_char_p),
    "pmoe_expert_bytes": ([_I, _I, _I], ctypes.c_size_t),
    "moe_router_topk": ([_P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_router_gemm_topk": ([_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_group_by_expert": ([_P, _I, _I, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P], _I),
    "moe_group_scratch_ints": ([_I, _I], ctypes.c_size_t),
    "expert_cache_create": ([ctypes.POINTER(pmoe_cache_desc), ctypes.POINTER(_P)], _I),
    "expert_cache_destroy": ([_P], None),
    "expert_cache_host_store": ([_P, _I, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)], _I),
    "expert_cache_load_expert": ([_P, _I, _I, _P, ctypes.c_size_t], _I),
    "expert_cache_reset": ([_P, _I], _I),
    "expert_cache_ensure_resident": ([_P, _I, _P, _I, _P, ctypes.POINTER(_I)], _I),
    "expert_cache_prefetch": ([_P, _I, _P, _I, _P], _I),
    "moe_paged_forward": ([_P, _I, _P, _I, _P, _P, _P, _P, _P], _I),
    "expert_cache_stats": ([_P, _I, ctypes.POINTER(pmoe_stats)], _I),
    "expert_cache_slot_table": ([_P, _I, _P, _P], _I),
    "expert_cache_read_slot": ([_P, _I, _I, _P, ctypes.c_size_t], _I),
    "expert_cache_set_timing": ([_P, _I], _I),
    "expert_cache_kernel_times": ([_P, ctypes.POINTER(pmoe_kernel_times)], _I),
    "moe_decode_forward_noalloc": ([_P, ctypes.c_size_t, _I, _P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P,
                                    _P], _I),
    "moe_paged_stack_forward": ([_P, _P, _I, _P, _P, _P, _P, _P], _I),
}
EXPORTED = tuple(_SIGS)


def load(path=LIB_PATH):
    """Load the library (building it first if sources are newer)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    from . import build as _build
    if _build.needs_build():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libpagedmoe.so not found at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = lib
    return lib


def _check(status, what):
    if status != PMOE_OK:
        raise PmoeError(status, what)


def _stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def pmoe_expert_bytes(fmt, H, I):
    return int(load().pmoe_expert_bytes(fmt, H, I))


def moe_router_topk(logits, top_k, renormalize=True, ids_out=None, w_out=None, stream=None):
    """logits: CUDA fp32 [T, E] -> (ids int32 [T, top_k], w fp32 [T, top_k])."""
    import torch
    lib = load()
    T, E = logits.shape
    assert logits.dtype == torch.float32 and logits.is_cuda and logits.is_contiguous()
    if ids_out is None:
        ids_out = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if w_out is None:
        w_out = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _check(lib.moe_router_topk(_ptr(logits), T, E, top_k, 1 if renormalize else 0, _ptr(ids_out), _ptr(w_out),
                               _stream_handle(stream)), "moe_router_topk")
    return ids_out, w_out


def moe_group_by_expert(ids, E, err_out=None, stream=None):
    """ids: CUDA int32 (any shape, flattened to P pairs) -> (counts [E], offs [E + 1],
    perm [P], pos [P]) int32; perm entries from offs[E] on (ids outside [0, E)) are
    undefined. err_out (CUDA int32 [1]) gets 1 ORed in for such an id."""
    import torch
    lib = load()
    assert ids.dtype == torch.int32 and ids.is_cuda and ids.is_contiguous()
    P = ids.numel()
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(P, 1), dtype=torch.int32, device=dev)[:P]
    pos = torch.empty(max(P, 1), dtype=torch.int32, device=dev)[:P]
    n_scratch = int(lib.moe_group_scratch_ints(P, E))
    scratch = torch.empty(n_scratch, dtype=torch.int32, device=dev) if n_scratch > 0 else None
    _check(lib.moe_group_by_expert(_ptr(ids), P, E, _ptr(counts), _ptr(offs), _ptr(perm), _ptr(pos), _ptr(scratch),
                                   n_scratch, _ptr(err_out), _stream_handle(stream)), "moe_group_by_expert")
    return counts, offs, perm, pos


def moe_router_gemm_topk(x, router_weight, top_k, renormalize=True, ids_out=None, w_out=None, logits_out=None,
                         stream=None):
    """x: CUDA bf16 [T, H], router_weight: CUDA bf16 [E, H] -> (ids int32 [T, top_k],
    w fp32 [T, top_k]); logits_out (fp32 [T, E]) is filled when given."""
    import torch
    lib = load()
    T, H = x.shape
    E = router_weight.shape[0]
    assert x.dtype == torch.bfloat16 and router_weight.dtype == torch.bfloat16 and router_weight.shape[1] == H
    assert x.is_cuda and x.is_contiguous() and router_weight.is_contiguous()
    if ids_out is None:
        ids_out = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if w_out is None:
        w_out = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    _check(lib.moe_router_gemm_topk(_ptr(x), _ptr(router_weight), T, H, E, top_k, 1 if renormalize else 0,
                                    _ptr(logits_out), _ptr(ids_out), _ptr(w_out), _stream_handle(stream)),
           "moe_router_gemm_topk")
    return ids_out, w_out


def moe_decode_forward_noalloc(experts, stride, E, top_k, H, I, fmt, x, ids, w, y=None, slot_of=None,
                               residual=None, err_out=None, n_slots=None, stream=None):
    """Decode MoE over experts already in device memory; allocates no device memory
    (the library uses a fixed static scratch). experts: CUDA uint8 tensor holding the
    expert slots `stride` bytes apart (n_slots defaults to all of them); x: bf16 [T, H];
    ids int32 / w fp32 [T, top_k]; slot_of: int32 [E] or None; err_out: int32 [1] that
    receives the call's device error bits, or None. Returns y."""
    import torch
    T = x.shape[0]
    assert experts.is_cuda and experts.dtype == torch.uint8 and experts.is_contiguous()
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous() and x.shape == (T, H)
    assert ids.is_cuda and ids.dtype == torch.int32 and ids.is_contiguous() and tuple(ids.shape) == (T, top_k)
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous() and tuple(w.shape) == (T, top_k)
    if slot_of is not None:
        assert slot_of.is_cuda and slot_of.dtype == torch.int32 and slot_of.is_contiguous() and slot_of.numel() == E
    if residual is not None:
        assert residual.is_cuda and residual.dtype == torch.bfloat16 and residual.is_contiguous()
        assert residual.shape == x.shape
    if err_out is not None:
        assert err_out.is_cuda and err_out.dtype == torch.int32 and err_out.numel() >= 1
    if n_slots is None:
        n_slots = experts.numel() // stride
    if y is None:
        y = torch.empty_like(x)
    assert y.is_cuda and y.dtype == torch.bfloat16 and y.is_contiguous() and y.shape == x.shape
    _check(load().moe_decode_forward_noalloc(_ptr(experts), stride, n_slots, _ptr(slot_of), E, top_k, H, I, fmt,
                                             _ptr(x), T, _ptr(ids), _ptr(w), _ptr(residual), _ptr(y), _ptr(err_out),
                                             _stream_handle(stream)), "moe_decode_forward_noalloc")
    return y


class ExpertCache:
    """Owns one pmoe_cache (expert_cache_create ... expert_cache_destroy)."""

    def __init__(self, num_experts, top_k, hidden, intermediate, num_slots, num_layers=1, fmt=PMOE_BF16,
                 max_tokens=8, pagein_mode=PMOE_PAGEIN_COPY_ENGINE, device=0):
        lib = load()
        self.desc = pmoe_cache_desc(num_experts, top_k, hidden, intermediate, num_slots, num_layers, fmt,
                                    max_tokens, pagein_mode, device)
        h = ctypes.c_void_p()
        _check(lib.expert_cache_create(ctypes.byref(self.desc), ctypes.byref(h)), "expert_cache_create")
        self.handle = h
        self.E, self.top_k, self.H, self.I, self.K = num_experts, top_k, hidden, intermediate, num_slots
        self.layers, self.fmt, self.max_tokens = num_layers, fmt, max_tokens
        self.expert_bytes = pmoe_expert_bytes(fmt, hidden, intermediate)

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            load().expert_cache_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- host store
    def host_store(self, layer):
        """numpy uint8 view [E, stride] of the layer's pinned store."""
        p = ctypes.c_void_p()
        stride = ctypes.c_size_t()
        _check(load().expert_cache_host_store(self.handle, layer, ctypes.byref(p), ctypes.byref(stride)),
               "expert_cache_host_store")
        buf = (ctypes.c_uint8 * (self.E * stride.value)).from_address(p.value)
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.E, stride.value)

    def load_layer(self, layer, experts):
        """experts: uint8 [E, expert_bytes] -> copied into the store."""
        view = self.host_store(layer)
        view[:, :self.expert_bytes] = experts

    def expert_cache_load_expert(self, layer, expert, data):
        data = np.ascontiguousarray(data, dtype=np.uint8)
        _check(load().expert_cache_load_expert(self.handle, layer, expert, data.ctypes.data_as(ctypes.c_void_p),
                                               data.size), "expert_cache_load_expert")

    def expert_cache_reset(self, layer=-1):
        _check(load().expert_cache_reset(self.handle, layer), "expert_cache_reset")

    def expert_cache_ensure_resident(self, layer, ids, stream=None):
        waves = ctypes.c_int(0)
        _check(load().expert_cache_ensure_resident(self.handle, layer, _ptr(ids), ids.numel(),
                                                   _stream_handle(stream), ctypes.byref(waves)),
               "expert_cache_ensure_resident")
        return waves.value

    def expert_cache_prefetch(self, layer, ids, stream=None):
        _check(load().expert_cache_prefetch(self.handle, layer, _ptr(ids), ids.numel(), _stream_handle(stream)),
               "expert_cache_prefetch")

    def moe_paged_forward(self, layer, x, ids, w, y=None, residual=None, stream=None):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        assert x.dtype == torch.bfloat16 and ids.dtype == torch.int32 and w.dtype == torch.float32
        _check(load().moe_paged_forward(self.handle, layer, _ptr(x), T, _ptr(ids), _ptr(w), _ptr(residual), _ptr(y),
                                        _stream_handle(stream)), "moe_paged_forward")
        return y

    def moe_paged_stack_forward(self, x, ids_all, w_all, y=None, work=None, stream=None):
        """All layers: h_{l+1} = h_l + moe_l(h_l). ids_all/w_all: [L, T, top_k] device."""
        import torch
        if y is None:
            y = torch.empty_like(x)
        if work is None and self.layers > 1:
            work = torch.empty_like(x)
        _check(load().moe_paged_stack_forward(self.handle, _ptr(x), x.shape[0], _ptr(ids_all), _ptr(w_all), _ptr(y),
                                              _ptr(work), _stream_handle(stream)), "moe_paged_stack_forward")
        return y

    def expert_cache_stats(self, layer=-1):
        s = pmoe_stats()
        _check(load().expert_cache_stats(self.handle, layer, ctypes.byref(s)), "expert_cache_stats")
        return {n: int(getattr(s, n)) for n, _ in pmoe_stats._fields_}

    def expert_cache_slot_table(self, layer):
        exp = np.empty(self.K, np.int32)
        lu = np.empty(self.K, np.int32)
        _check(load().expert_cache_slot_table(self.handle, layer, exp.ctypes.data_as(ctypes.c_void_p),
                                              lu.ctypes.data_as(ctypes.c_void_p)), "expert_cache_slot_table")
        return exp, lu

    def expert_cache_read_slot(self, layer, slot):
        out = np.empty(self.expert_bytes, np.uint8)
        _check(load().expert_cache_read_slot(self.handle, layer, slot, out.ctypes.data_as(ctypes.c_void_p),
                                             out.size), "expert_cache_read_slot")
        return out

    def expert_cache_set_timing(self, enable=True):
        _check(load().expert_cache_set_timing(self.handle, 1 if enable else 0), "expert_cache_set_timing")

    def expert_cache_kernel_times(self):
        kt = pmoe_kernel_times()
        _check(load().expert_cache_kernel_times(self.handle, ctypes.byref(kt)), "expert_cache_kernel_times")
        return {name: {"ms": kt.ms[i], "launches": int(kt.launches[i])} for i, name in enumerate(KERNEL_CLASSES)} | \
            {"copies": int(kt.copies)}
