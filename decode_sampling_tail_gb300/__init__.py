"""GB300-native decode sampling tail: final RMSNorm -> bf16 lm_head -> global top-k -> sampler.

Thin ctypes binding of ``libtail.so`` (C ABI declared in ``include/tail.h``).
The functions below only marshal arguments: every step of the tail runs in
the library's CUDA kernels.  There is no CPU fallback: importing works without
the library, but creating a handle raises ``TailLibraryMissing`` when
``libtail.so`` has not been built (``python -m decode_sampling_tail_gb300.build``
or ``__graft_entry__.build()``).

The operation follows "GPT-OSS Tail Chunked Megakernel Kernel API Reference"
(function gpt_oss_tail_chunked_megakernel) on one GPU holding the whole
vocabulary.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtail.so")

TAIL_F32, TAIL_F16, TAIL_BF16 = 0, 1, 2
TAIL_OK = 0
TAIL_ERR_INVALID_ARG = -1
TAIL_ERR_UNSUPPORTED = -2
TAIL_ERR_CUDA = -3
TAIL_ERR_OOM = -4
TAIL_ERR_DEVICE = -5
# tail_path: which lm_head serves which batch sizes ("gemv": mma.sync kernel up to 8 rows,
# "tensor": tensor-core path for every batch, "auto": "tensor" for narrow vocabularies,
# "small": one launch for every batch of a small problem, bound by latency)
PATHS = {"auto": 0, "gemv": 1, "tensor": 2, "small": 3}
TC_ALL_ROWS_MAX_V = 131072

EXPORTS = ("tail_create", "tail_run", "tail_run_ex", "tail_run_host", "tail_check", "tail_get_info",
           "tail_destroy", "tail_status_string", "tail_profile_enable", "tail_profile_read",
           "tail_set_wait_limit", "tail_debug_drop_stage", "tail_last_error", "tail_run_noalloc",
           "tail_merge_shards", "tail_run_moe", "tail_tap_shape", "tail_run_taps", "tail_prepare_weight")
KERNELS = ("rms_rows", "lm_head", "merge")


class TailLibraryMissing(RuntimeError):
    pass


class TailError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status in (TAIL_ERR_CUDA, TAIL_ERR_OOM):
            try:
                detail = " [" + lib().tail_last_error().decode() + "]"
            except TailLibraryMissing:
                pass
        super().__init__(f"{what}: {status_string(status)} ({status}){detail}")


class tail_config(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("hidden_actual", ctypes.c_int32), ("V", ctypes.c_int32),
                ("k", ctypes.c_int32), ("gbs_max", ctypes.c_int32), ("eps", ctypes.c_float),
                ("hidden_dtype", ctypes.c_int32), ("zero_interleaved_pad", ctypes.c_int32),
                ("deferred_rms", ctypes.c_int32), ("path", ctypes.c_int32)]


class tail_info(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("nslab", ctypes.c_int32), ("merge_groups", ctypes.c_int32),
                ("lmhead_path", ctypes.c_int32), ("rows_per_pass", ctypes.c_int32),
                ("kernels_per_run", ctypes.c_int32), ("scratch_bytes", ctypes.c_int64),
                ("tc_min_rows", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def lib(path: str | None = None):
    """Loads libtail.so (raises TailLibraryMissing if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise TailLibraryMissing(f"{p} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(p)
        P, i32 = ctypes.c_void_p, ctypes.c_int32
        L.tail_create.argtypes = [ctypes.POINTER(tail_config), ctypes.c_int, ctypes.POINTER(P)]
        L.tail_create.restype = ctypes.c_int
        L.tail_run.argtypes = [P, P, P, P, P, i32, i32, P, P, P]
        L.tail_run.restype = ctypes.c_int
        L.tail_run_ex.argtypes = [P, P, P, P, P, i32, i32, P, P, P, P, P]
        L.tail_run_ex.restype = ctypes.c_int
        L.tail_run_moe.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, i32, i32, P, P, P, P, P, P]
        L.tail_run_moe.restype = ctypes.c_int
        L.tail_tap_shape.argtypes = [P, i32, P, P, P, P]
        L.tail_tap_shape.restype = ctypes.c_int
        L.tail_run_taps.argtypes = [P, P, P, P, P, i32, i32, P, P, P, P, P, P, P, P, P]
        L.tail_run_taps.restype = ctypes.c_int
        L.tail_prepare_weight.argtypes = [P, P, P]
        L.tail_prepare_weight.restype = ctypes.c_int
        L.tail_run_host.argtypes = [P, P, P, P, P, i32, i32, P, P, P]
        L.tail_run_host.restype = ctypes.c_int
        L.tail_run_noalloc.argtypes = [ctypes.POINTER(tail_config), P, P, P, P, i32, i32, P, P, P, P]
        L.tail_run_noalloc.restype = ctypes.c_int
        L.tail_merge_shards.argtypes = [i32, i32, i32, i32, P, P, ctypes.POINTER(i32), P, i32, P, P, P, P]
        L.tail_merge_shards.restype = ctypes.c_int
        L.tail_check.argtypes = [P]
        L.tail_check.restype = ctypes.c_int
        L.tail_get_info.argtypes = [P, ctypes.POINTER(tail_info)]
        L.tail_get_info.restype = ctypes.c_int
        L.tail_destroy.argtypes = [P]
        L.tail_destroy.restype = None
        L.tail_profile_enable.argtypes = [P, ctypes.c_int]
        L.tail_profile_enable.restype = ctypes.c_int
        L.tail_profile_read.argtypes = [P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int32)]
        L.tail_profile_read.restype = ctypes.c_int
        L.tail_set_wait_limit.argtypes = [P, ctypes.c_uint64]
        L.tail_set_wait_limit.restype = ctypes.c_int
        L.tail_debug_drop_stage.argtypes = [P, ctypes.c_int32]
        L.tail_debug_drop_stage.restype = ctypes.c_int
        L.tail_last_error.argtypes = []
        L.tail_last_error.restype = ctypes.c_char_p
        L.tail_status_string.argtypes = [ctypes.c_int]
        L.tail_status_string.restype = ctypes.c_char_p
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return lib().tail_status_string(status).decode()
    except TailLibraryMissing:
        return "library missing"


# ------------------------------------------------------------------ raw C-ABI mirrors (pointers as ints)

def tail_create(cfg: tail_config, device: int = 0) -> int:
    h = ctypes.c_void_p()
    rc = lib().tail_create(ctypes.byref(cfg), device, ctypes.byref(h))
    if rc != TAIL_OK:
        raise TailError(rc, "tail_create")
    return h.value


def tail_run(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt, stream) -> int:
    return lib().tail_run(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt, stream)


def tail_run_ex(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt,
                out_topk_vals_opt, out_topk_idx_opt, stream) -> int:
    return lib().tail_run_ex(h, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens, out_logits_opt,
                             out_topk_vals_opt, out_topk_idx_opt, stream)


def tail_run_moe(h, residual, slots, slot_dtype, nslots, n_routed, slot_w, gamma, w_t, params, n_param_cols, gbs,
                 out_tokens, out_logits_opt, out_topk_vals_opt, out_topk_idx_opt, out_hidden_opt, stream) -> int:
    return lib().tail_run_moe(h, residual, slots, slot_dtype, nslots, n_routed, slot_w, gamma, w_t, params,
                              n_param_cols, gbs, out_tokens, out_logits_opt, out_topk_vals_opt, out_topk_idx_opt,
                              out_hidden_opt, stream)


def tail_run_host(h, hidden_host, gamma, w_t, params_host, n_param_cols, gbs, out_tokens_host,
                  out_logits_host_opt, stream) -> int:
    return lib().tail_run_host(h, hidden_host, gamma, w_t, params_host, n_param_cols, gbs, out_tokens_host,
                               out_logits_host_opt, stream)


def tail_run_noalloc(cfg: tail_config, hidden, gamma, w_t, params, n_param_cols, gbs, out_tokens,
                     out_logits_opt, out_status_opt, stream) -> int:
    return lib().tail_run_noalloc(ctypes.byref(cfg), hidden, gamma, w_t, params, n_param_cols, gbs,
                                  out_tokens, out_logits_opt, out_status_opt, stream)


def tail_merge_shards(nshard, k_in, k, gbs, cand_vals, cand_idx, shard_offsets, params, n_param_cols, out_tokens,
                      out_topk_vals_opt, out_topk_idx_opt, stream) -> int:
    offs = (ctypes.c_int32 * len(shard_offsets))(*[int(o) for o in shard_offsets])
    return lib().tail_merge_shards(nshard, k_in, k, gbs, cand_vals, cand_idx, offs, params, n_param_cols,
                                   out_tokens, out_topk_vals_opt, out_topk_idx_opt, stream)


def tail_check(h) -> int:
    return lib().tail_check(h)


def tail_get_info(h) -> tail_info:
    info = tail_info()
    rc = lib().tail_get_info(h, ctypes.byref(info))
    if rc != TAIL_OK:
        raise TailError(rc, "tail_get_info")
    return info


def tail_profile_enable(h, enable: bool) -> int:
    return lib().tail_profile_enable(h, int(enable))


def tail_profile_read(h):
    """Returns ({kernel name: summed ms}, passes recorded)."""
    ms = (ctypes.c_float * len(KERNELS))()
    n = ctypes.c_int32()
    rc = lib().tail_profile_read(h, ms, ctypes.byref(n))
    if rc != TAIL_OK:
        raise TailError(rc, "tail_profile_read")
    return dict(zip(KERNELS, list(ms))), n.value


def tail_set_wait_limit(h, ns: int) -> int:
    return lib().tail_set_wait_limit(h, ctypes.c_uint64(ns))


def tail_debug_drop_stage(h, iteration: int) -> int:
    return lib().tail_debug_drop_stage(h, iteration)


def tail_destroy(h) -> None:
    if h:
        lib().tail_destroy(h)


# ------------------------------------------------------------------ torch convenience wrapper

_DTYPES = {"f32": TAIL_F32, "f16": TAIL_F16, "bf16": TAIL_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def run_noalloc(hidden, gamma, w_t, params=None, out_tokens=None, out_logits=None, out_status=None, *,
                k: int = 256, hidden_actual: int = 0, eps: float = 1e-5, hidden_dtype: str = "bf16",
                zero_interleaved_pad: bool = True, deferred_rms: bool = True, stream=None):
    """tail_run_noalloc on the current device with torch CUDA tensors (see ``Tail`` for their layout).

    No handle and no device allocation: the library's static per-device scratch is used, so
    calls whose kernels may overlap must be serialised by the caller.  ``out_status`` is an
    optional int32 CUDA tensor of one element receiving the kernels' error word.
    """
    gbs, H = int(hidden.shape[0]), int(hidden.shape[1])
    V = int(w_t.shape[1])
    cfg = tail_config(H, hidden_actual, V, k, max(gbs, 1), eps, _DTYPES[hidden_dtype],
                      int(zero_interleaved_pad), int(deferred_rms))
    ncols = int(params.shape[1]) if params is not None else 4
    rc = tail_run_noalloc(cfg, _ptr(hidden), _ptr(gamma), _ptr(w_t), _ptr(params), ncols, gbs,
                          _ptr(out_tokens), _ptr(out_logits), _ptr(out_status),
                          _stream_ptr(stream, hidden.device))
    if rc == TAIL_ERR_UNSUPPORTED:
        raise TailError(rc, "tail_run_noalloc [" + lib().tail_last_error().decode() + "]")
    if rc != TAIL_OK:
        raise TailError(rc, "tail_run_noalloc")
    return out_tokens


class Tail:
    """A tail handle bound to one device; tensors are torch CUDA tensors.

    ``hidden`` is [gbs, H] (float32, float16 or bfloat16 matching ``hidden_dtype``;
    uint16/int16 bit patterns are accepted for the 16-bit types), ``gamma`` [H]
    float32, ``w_t`` [H, V] bfloat16 (or its int16 bits), ``params`` [gbs, 3|4]
    float32 or None.  ``path`` is a key of ``PATHS``.
    """

    def __init__(self, H: int, V: int, k: int = 256, gbs_max: int = 64, *, hidden_actual: int = 0,
                 eps: float = 1e-5, hidden_dtype: str = "bf16", zero_interleaved_pad: bool = True,
                 deferred_rms: bool = True, path: str = "auto", device: int = 0):
        self.cfg = tail_config(H, hidden_actual, V, k, gbs_max, eps, _DTYPES[hidden_dtype],
                               int(zero_interleaved_pad), int(deferred_rms), PATHS[path])
        self.device = device
        self.h = tail_create(self.cfg, device)
        self.info = tail_get_info(self.h)

    def close(self):
        if self.h:
            tail_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _stream(self, stream):
        if stream is None:
            import torch
            stream = torch.cuda.current_stream(self.device)
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))

    def run(self, hidden, gamma, w_t, params=None, out_tokens=None, out_logits=None, out_topk_vals=None,
            out_topk_idx=None, stream=None):
        gbs = int(hidden.shape[0])
        ncols = int(params.shape[1]) if params is not None else 4
        rc = tail_run_ex(self.h, _ptr(hidden), _ptr(gamma), _ptr(w_t), _ptr(params), ncols, gbs,
                         _ptr(out_tokens), _ptr(out_logits), _ptr(out_topk_vals), _ptr(out_topk_idx),
                         self._stream(stream))
        if rc != TAIL_OK:
            raise TailError(rc, "tail_run_ex")
        return out_tokens

    def prepare_weight(self, w_t, stream=None):
        """tail_prepare_weight: the tensor-core path's copy of w_t (None frees it)."""
        rc = lib().tail_prepare_weight(self.h, _ptr(w_t), self._stream(stream))
        if rc != TAIL_OK:
            raise TailError(rc, "tail_prepare_weight")
        self.info = tail_get_info(self.h)

    def run_moe(self, residual, slots, slot_w, gamma, w_t, params=None, out_tokens=None, out_logits=None,
                out_topk_vals=None, out_topk_idx=None, out_hidden=None, n_routed=None, stream=None):
        """The tail fused with its producer (tail_run_moe): residual [gbs, H] bf16, slots [gbs, S, H]
        float32 or bf16, slot_w [gbs, S] float32, n_routed the leading slots of the routed chain (None:
        all S; the rest are shared slots, summed apart); out_hidden [gbs, H] bf16 receives the combined h."""
        import torch
        gbs = int(residual.shape[0])
        S = int(slots.shape[1]) if slots is not None else 0
        nr = S if n_routed is None else int(n_routed)
        sd = TAIL_F32 if slots is None or slots.dtype == torch.float32 else TAIL_BF16
        ncols = int(params.shape[1]) if params is not None else 4
        rc = tail_run_moe(self.h, _ptr(residual), _ptr(slots), sd, S, nr, _ptr(slot_w), _ptr(gamma), _ptr(w_t),
                          _ptr(params), ncols, gbs, _ptr(out_tokens), _ptr(out_logits), _ptr(out_topk_vals),
                          _ptr(out_topk_idx), _ptr(out_hidden), self._stream(stream))
        if rc != TAIL_OK:
            raise TailError(rc, "tail_run_moe")
        return out_tokens

    def tap_shape(self, gbs):
        """(kind, n_chunks, cap, chunk_lo) of tail_tap_shape: kind 1 = slabs, 2 = tiles; chunk_lo a list of
        n_chunks + 1 vocabulary ids (the chunks' first ids, then V)."""
        kind, n, cap = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        rc = lib().tail_tap_shape(self.h, gbs, ctypes.byref(kind), ctypes.byref(n), ctypes.byref(cap), None)
        if rc != TAIL_OK:
            raise TailError(rc, "tail_tap_shape")
        lo = (ctypes.c_int32 * (n.value + 1))()
        lib().tail_tap_shape(self.h, gbs, ctypes.byref(kind), ctypes.byref(n), ctypes.byref(cap), lo)
        return kind.value, n.value, cap.value, list(lo)

    def run_taps(self, hidden, gamma, w_t, params=None, out_tokens=None, out_logits=None, out_topk_vals=None,
                 out_topk_idx=None, stream=None):
        """tail_run_taps: the run plus its stage-1 taps, returned as torch tensors
        (vals [gbs, n, cap] float32, idx [gbs, n, cap] int32, count [gbs, n] int32, bound [gbs, n] float32)."""
        import torch
        gbs = int(hidden.shape[0])
        _, n, cap, _ = self.tap_shape(gbs)
        dev = hidden.device
        vals = torch.empty((gbs, n, cap), dtype=torch.float32, device=dev)
        idx = torch.empty((gbs, n, cap), dtype=torch.int32, device=dev)
        count = torch.empty((gbs, n), dtype=torch.int32, device=dev)
        bound = torch.empty((gbs, n), dtype=torch.float32, device=dev)
        ncols = int(params.shape[1]) if params is not None else 4
        rc = lib().tail_run_taps(self.h, _ptr(hidden), _ptr(gamma), _ptr(w_t), _ptr(params), ncols, gbs,
                                 _ptr(out_tokens), _ptr(out_logits), _ptr(out_topk_vals), _ptr(out_topk_idx),
                                 _ptr(vals), _ptr(idx), _ptr(count), _ptr(bound), self._stream(stream))
        if rc != TAIL_OK:
            raise TailError(rc, "tail_run_taps")
        return vals, idx, count, bound

    def run_host(self, hidden_host, gamma, w_t, params_host=None, out_tokens_host=None,
                 out_logits_host=None, stream=None):
        """hidden_host / params_host / outputs are host (ideally pinned) tensors or numpy arrays."""
        def hp(x):
            if x is None:
                return None
            if hasattr(x, "data_ptr"):
                return ctypes.c_void_p(x.data_ptr())
            return x.ctypes.data_as(ctypes.c_void_p)
        gbs = int(hidden_host.shape[0])
        ncols = int(params_host.shape[1]) if params_host is not None else 4
        rc = tail_run_host(self.h, hp(hidden_host), _ptr(gamma), _ptr(w_t), hp(params_host), ncols, gbs,
                           hp(out_tokens_host), hp(out_logits_host), self._stream(stream))
        if rc != TAIL_OK:
            raise TailError(rc, "tail_run_host")
        return out_tokens_host

    def check(self):
        rc = tail_check(self.h)
        if rc != TAIL_OK:
            raise TailError(rc, "tail_check")


def merge_shards(cand_vals, cand_idx, shard_offsets, k, params=None, out_tokens=None, out_topk_vals=None,
                 out_topk_idx=None, stream=None):
    """tail_merge_shards with torch CUDA tensors: cand_vals [nshard, gbs, k_in] float32, cand_idx the same
    shape int32 (ids within each shard), shard_offsets a sequence of each shard's first global id."""
    nshard, gbs, k_in = (int(d) for d in cand_vals.shape)
    ncols = int(params.shape[1]) if params is not None else 4
    rc = tail_merge_shards(nshard, k_in, k, gbs, _ptr(cand_vals), _ptr(cand_idx), list(shard_offsets),
                           _ptr(params), ncols, _ptr(out_tokens), _ptr(out_topk_vals), _ptr(out_topk_idx),
                           _stream_ptr(stream, cand_vals.device))
    if rc == TAIL_ERR_UNSUPPORTED:
        raise TailError(rc, "tail_merge_shards [" + lib().tail_last_error().decode() + "]")
    if rc != TAIL_OK:
        raise TailError(rc, "tail_merge_shards")
    return out_tokens
