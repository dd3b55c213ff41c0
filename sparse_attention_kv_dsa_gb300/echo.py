"""ctypes binding of libecho.so (include/echo.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels; PyTorch provides the
device memory, the pinned host memory and the current stream.  The binding raises
if the library has not been built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

# ---------------------------------------------------------------- constants --
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_POOL_EXHAUSTED, ERR_HOST_INDEX, ERR_STAGING = range(8)
ERR_SCRATCH_LIMIT = 8
ERR_NOT_RESIDENT = 9
MLA_NOALLOC_SCRATCH_BYTES = 32 << 20
PF_DEFER_CAP = 1            # echo_index_prefetch flag: exact cap restored by echo_topk_prefetch
F32, BF16, E4M3 = 0, 1, 2
KV_WIDTH, V_WIDTH = 576, 512
CTR_STEP, CTR_N_FREE, CTR_STATUS, CTR_NEED, CTR_CURSOR, CTR_EVICT_M = 0, 1, 2, 3, 4, 5
CTR_HITS, CTR_STAGED_HITS, CTR_MISSES, CTR_EVICTED, CTR_STAGED, CTR_WB_EVICTED, CTR_BOUND, CTR_QUALIFIED = range(8, 16)
NUM_COUNTERS = 32
PENDING_LIST_MIN_SLOTS = 14080  # ECHO_PENDING_LIST_MIN_SLOTS: pools that keep the pending victim list

STATUS_NAMES = {OK: "OK", ERR_INVALID_ARG: "INVALID_ARG", ERR_UNSUPPORTED: "UNSUPPORTED", ERR_CUDA: "CUDA",
                ERR_TIMEOUT: "TIMEOUT", ERR_POOL_EXHAUSTED: "POOL_EXHAUSTED", ERR_HOST_INDEX: "HOST_INDEX",
                ERR_STAGING: "STAGING", ERR_SCRATCH_LIMIT: "SCRATCH_LIMIT", ERR_NOT_RESIDENT: "NOT_RESIDENT"}


class EchoError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        super().__init__(f"echo {where}: {STATUS_NAMES.get(self.code, self.code)}")


class CacheLayerT(ctypes.Structure):
    _fields_ = [("n_gpu", ctypes.c_int32), ("n_host", ctypes.c_int32),
                ("host2gpu", ctypes.c_void_p), ("gpu2host", ctypes.c_void_p), ("priority", ctypes.c_void_p),
                ("index_buf", ctypes.c_void_p), ("free_map", ctypes.c_void_p), ("counters", ctypes.c_void_p),
                ("gpu_kv", ctypes.c_void_p), ("host_kv", ctypes.c_void_p), ("kv_dtype", ctypes.c_int32),
                ("pf_new_rows", ctypes.c_void_p), ("pf_pred_err", ctypes.c_void_p), ("cap_slack", ctypes.c_int32),
                ("block_tokens", ctypes.c_int32), ("row_elems", ctypes.c_int32)]


class StepArgsT(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("host_base", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
                ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("Lmax", ctypes.c_int32), ("idx_dtype", ctypes.c_int32),
                ("q_idx", ctypes.c_void_p), ("w_idx", ctypes.c_void_p), ("idx_k", ctypes.c_void_p),
                ("new_ik", ctypes.c_void_p), ("new_kv", ctypes.c_void_p), ("theta", ctypes.c_void_p),
                ("alpha", ctypes.c_float), ("k", ctypes.c_int32), ("prefetch", ctypes.c_int32),
                ("cap_max", ctypes.c_int32), ("cap_div", ctypes.c_int32), ("cap", ctypes.c_void_p),
                ("scores", ctypes.c_void_p), ("pf_list", ctypes.c_void_p), ("pf_count", ctypes.c_void_p),
                ("stage_kv", ctypes.c_void_p), ("sel", ctypes.c_void_p), ("kth", ctypes.c_void_p),
                ("miss_list", ctypes.c_void_p), ("n_miss", ctypes.c_void_p), ("slot_idx", ctypes.c_void_p),
                ("Hq", ctypes.c_int32), ("q_mla", ctypes.c_void_p), ("scale", ctypes.c_float),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("mla_workspace", ctypes.c_void_p),
                ("mla_workspace_bytes", ctypes.c_size_t), ("index_events", ctypes.c_void_p * 2)]


HOST_POOL_MAX_RANGES = 1024    # ECHO_HOST_POOL_MAX_RANGES


class HostPoolT(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("n_layers", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("rows_per_layer", ctypes.c_int64), ("rows_in_use", ctypes.c_int64), ("n_free", ctypes.c_int32),
                ("free_first", ctypes.c_int64 * HOST_POOL_MAX_RANGES),
                ("free_rows", ctypes.c_int64 * HOST_POOL_MAX_RANGES)]


# Declared signatures: name -> (restype, argtypes).  P = pointer, I = int32.
_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "echo_cache_metadata_bytes": (_S, [ctypes.c_int64, ctypes.c_int64]),
    "echo_host_device_pointer": (_I, [_P, ctypes.POINTER(ctypes.c_void_p)]),
    "echo_device_sm_count": (_I, []),
    "echo_cache_reset": (_I, [_P, _P]),
    "echo_cache_writeback": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _P]),
    "echo_cache_reserve": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "echo_index_prefetch": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _P]),
    "echo_topk": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _F, _P]),
    "echo_topk_prefetch": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _F, _P, _I, _P, _P, _P, _P, _P, _P]),
    "echo_cache_evict": (_I, [_P, _P, _P]),
    "echo_cache_alloc": (_I, [_P, _P, _P, _I, _P, _P]),
    "echo_cache_recall": (_I, [_P, _P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P]),
    "echo_sparse_mla_workspace_bytes": (_S, [_I, _I, _I]),
    "echo_sparse_mla_decode": (_I, [_P, _P, _I, _I, _P, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "echo_abi_struct_sizes": (None, [_P]),
    "echo_sparse_gqa_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "echo_sparse_gqa_decode": (_I, [_P, _P, _I, _I, _P, _I, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "echo_sparse_mla_decode_noalloc": (_I, [_P, _P, _I, _I, _P, _I, _I, _I, _F, _P, _P, _P]),
    "echo_decode_layer_step": (_I, [_P, _P, _P]),
    "echo_prefill_index": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "echo_prefill_candidates": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "echo_mark_tokens": (_I, [_P, _I, _I, _P, _I, _P]),
    "echo_token_list": (_I, [_P, _I, _P, _I, _P, _P]),
    "echo_translate_slots": (_I, [_P, _P, _I, _I, _P, _I, _P, _P]),
    "echo_block_scores": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "echo_expand_block_slots": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "echo_host_pool_bytes": (_S, [_I, ctypes.c_int64, _I]),
    "echo_host_pool_init": (_I, [_P, _P, _I, ctypes.c_int64, _I]),
    "echo_host_pool_alloc": (_I, [_P, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]),
    "echo_host_pool_free": (_I, [_P, ctypes.c_int64, ctypes.c_int64]),
    "echo_host_pool_layer": (_I, [_P, _I, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p)]),
    "echo_cache_status": (_I, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "echo_cache_read_counters": (_I, [_P, ctypes.POINTER(ctypes.c_int32)]),
}

_LIB = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libecho.so (built in-tree).  Raises if it is missing."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: run `python -m sparse_attention_kv_dsa_gb300.build` "
                               "(or __graft_entry__.build()); there is no fallback path")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def check(code: int, where: str = "") -> None:
    if int(code) != OK:
        raise EchoError(code, where)


def ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def dtype_code(dt: torch.dtype) -> int:
    return {torch.float32: F32, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3, torch.uint8: E4M3}[dt]


def metadata_bytes(n_host: int, n_gpu: int) -> int:
    return int(lib().echo_cache_metadata_bytes(n_host, n_gpu))


def host_device_pointer(t: torch.Tensor) -> int:
    out = ctypes.c_void_p()
    check(lib().echo_host_device_pointer(t.data_ptr(), ctypes.byref(out)), "host_device_pointer")
    return int(out.value)


# ------------------------------------------------------------ layer cache ----
class LayerCache:
    """One layer's GPU cache: device metadata tensors, the GPU KV pool and the
    pinned host pool, described to the library by an echo_cache_layer_t."""

    def __init__(self, n_gpu: int, n_host: int, kv_dtype=torch.bfloat16, device="cuda", host_kv=None,
                 block_tokens: int = 1, row_elems: int = KV_WIDTH):
        """n_gpu / n_host count slots and host indices: tokens, or blocks of block_tokens
        tokens (then the pools hold n * block_tokens token rows).  A token row has
        row_elems values: the 576-wide MLA latent, or e.g. one KV head's key and value."""
        dev = torch.device(device)
        self.n_gpu, self.n_host, self.kv_dtype = int(n_gpu), int(n_host), kv_dtype
        self.block_tokens = T = max(int(block_tokens), 1)
        self.row_elems = W = int(row_elems)
        i32 = torch.int32
        self.host2gpu = torch.empty(n_host, dtype=i32, device=dev)
        self.gpu2host = torch.empty(n_gpu, dtype=i32, device=dev)
        self.priority = torch.empty(n_gpu, dtype=i32, device=dev)
        self.index_buf = torch.empty(n_gpu, dtype=i32, device=dev)
        self.free_map = torch.empty(n_gpu, dtype=torch.uint8, device=dev)
        self.counters = torch.zeros(NUM_COUNTERS, dtype=i32, device=dev)
        self.gpu_kv = torch.zeros(n_gpu * T, W, dtype=kv_dtype, device=dev)
        if host_kv is None:
            host_kv = torch.zeros(n_host * T, W, dtype=kv_dtype, pin_memory=True)
        assert host_kv.is_pinned() and host_kv.shape == (n_host * T, W) and host_kv.dtype == kv_dtype
        self.host_kv = host_kv
        self.host_kv_dev = host_device_pointer(host_kv)
        self.struct = CacheLayerT(self.n_gpu, self.n_host, ptr(self.host2gpu), ptr(self.gpu2host),
                                  ptr(self.priority), ptr(self.index_buf), ptr(self.free_map), ptr(self.counters),
                                  ptr(self.gpu_kv), self.host_kv_dev, dtype_code(kv_dtype))
        self.struct.block_tokens = T if T > 1 else 0
        self.struct.row_elems = W if W != KV_WIDTH else 0

    @property
    def ref(self):
        return ctypes.byref(self.struct)

    def reset(self, stream=None):
        check(lib().echo_cache_reset(self.ref, stream_handle(stream)), "cache_reset")

    def status(self) -> int:
        out = ctypes.c_int32()
        check(lib().echo_cache_status(self.ref, ctypes.byref(out)), "cache_status")
        return int(out.value)

    def read_counters(self) -> list:
        arr = (ctypes.c_int32 * NUM_COUNTERS)()
        check(lib().echo_cache_read_counters(self.ref, arr), "read_counters")
        return list(arr)

    def enable_adaptive_cap(self, B: int, slack: int) -> None:
        """Per-request state of the adaptive prefetch cap (no observation yet)."""
        dev = self.host2gpu.device
        self.pf_new_rows = torch.full((B,), -1, dtype=torch.int32, device=dev)
        self.pf_pred_err = torch.zeros(B, dtype=torch.float32, device=dev)
        self.struct.pf_new_rows, self.struct.pf_pred_err = ptr(self.pf_new_rows), ptr(self.pf_pred_err)
        self.struct.cap_slack = int(slack)

    def metadata_tensors(self):
        return (self.host2gpu, self.gpu2host, self.priority, self.index_buf, self.free_map)


# ------------------------------------------------------------- entry points --
def cache_writeback(layer: LayerCache, new_kv, new_ik, idx_k, host_base, seq_len, stream=None):
    B, D = new_ik.shape
    Lmax = idx_k.shape[1]
    check(lib().echo_cache_writeback(layer.ref, ptr(new_kv), ptr(new_ik), ptr(idx_k), D, Lmax,
                                     dtype_code(idx_k.dtype), ptr(host_base), ptr(seq_len), B,
                                     stream_handle(stream)), "cache_writeback")


def cache_reserve(layer: LayerCache, seq_len, cap_max: int, cap_div: int, cap, pf_count, stream=None):
    check(lib().echo_cache_reserve(layer.ref, ptr(seq_len), seq_len.shape[0], cap_max, cap_div, ptr(cap),
                                   ptr(pf_count), stream_handle(stream)), "cache_reserve")


def index_prefetch(q, w, idx_k, seq_len, theta, scores, *, layer: LayerCache | None = None, cap=None,
                   cap_max: int = 0, host_base=None, pf_list=None, pf_count=None, stage_kv=None,
                   defer_cap: bool = False, stream=None):
    B, H, D = q.shape
    Lmax = idx_k.shape[1]
    check(lib().echo_index_prefetch(ptr(q), ptr(w), ptr(idx_k), ptr(seq_len), B, H, D, Lmax, dtype_code(q.dtype),
                                    ptr(theta), ptr(cap), cap_max, ptr(host_base),
                                    layer.ref if layer is not None else None, ptr(scores), ptr(pf_list),
                                    ptr(pf_count), ptr(stage_kv), PF_DEFER_CAP if defer_cap else 0,
                                    stream_handle(stream)), "index_prefetch")


def topk(scores, seq_len, k: int, out_idx, kth, theta, alpha: float = 0.5, stream=None):
    B, Lmax = scores.shape
    check(lib().echo_topk(ptr(scores), ptr(seq_len), B, Lmax, k, ptr(out_idx), ptr(kth), ptr(theta), alpha,
                          stream_handle(stream)), "topk")


def topk_prefetch(scores, seq_len, k: int, out_idx, kth, theta, alpha: float, *, layer: LayerCache, cap,
                  cap_max: int, host_base, pf_list, pf_count, stage_kv, stream=None):
    """Top-k plus the exact prefetch cap deferred by index_prefetch(defer_cap=True)."""
    B, Lmax = scores.shape
    check(lib().echo_topk_prefetch(ptr(scores), ptr(seq_len), B, Lmax, k, ptr(out_idx), ptr(kth), ptr(theta), alpha,
                                   ptr(cap), cap_max, ptr(host_base), layer.ref, ptr(pf_list), ptr(pf_count),
                                   ptr(stage_kv), stream_handle(stream)), "topk_prefetch")


def cache_evict(layer: LayerCache, n_needed, stream=None):
    check(lib().echo_cache_evict(layer.ref, ptr(n_needed), stream_handle(stream)), "cache_evict")


def cache_alloc(layer: LayerCache, host_idx, n, out_slot, stream=None):
    check(lib().echo_cache_alloc(layer.ref, ptr(host_idx), ptr(n), host_idx.shape[0], ptr(out_slot),
                                 stream_handle(stream)), "cache_alloc")


def cache_recall(layer: LayerCache, sel, host_base, miss_list, n_miss, slot_idx, *, pf_list=None, pf_count=None,
                 cap_max: int = 0, stage_kv=None, stream=None):
    B, k = sel.shape
    check(lib().echo_cache_recall(layer.ref, ptr(sel), ptr(host_base), B, k, ptr(pf_list), ptr(pf_count), cap_max,
                                  ptr(stage_kv), ptr(miss_list), ptr(n_miss), ptr(slot_idx),
                                  stream_handle(stream)), "cache_recall")


def mla_workspace_bytes(B: int, Hq: int, k: int) -> int:
    return int(lib().echo_sparse_mla_workspace_bytes(B, Hq, k))


def sparse_mla_decode(q, kv, slot_idx, scale: float, out, lse, workspace, stream=None):
    B, Hq, _ = q.shape
    k = slot_idx.shape[1]
    check(lib().echo_sparse_mla_decode(ptr(q), ptr(kv), kv.shape[0], dtype_code(q.dtype), ptr(slot_idx), B, Hq, k,
                                       scale, ptr(out), ptr(lse), ptr(workspace),
                                       workspace.numel() * workspace.element_size(), stream_handle(stream)),
          "sparse_mla_decode")


def gqa_workspace_bytes(NG: int, G: int, d: int, k: int) -> int:
    return int(lib().echo_sparse_gqa_workspace_bytes(NG, G, d, k))


def sparse_gqa_decode(q, kv, slot_idx, scale: float, out, lse, workspace=None, stream=None):
    """q [NG,G,d] (one group = one request's KV head), kv [rows,2d], slot_idx [NG,k]."""
    NG, G, d = q.shape
    k = slot_idx.shape[1]
    ws = ptr(workspace) if workspace is not None else None
    nb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().echo_sparse_gqa_decode(ptr(q), ptr(kv), kv.shape[0], dtype_code(q.dtype), ptr(slot_idx), NG, G, d,
                                       k, scale, ptr(out), ptr(lse), ws, nb, stream_handle(stream)),
          "sparse_gqa_decode")


def decode_layer_step(layer: LayerCache, args: StepArgsT, stream=None):
    check(lib().echo_decode_layer_step(layer.ref, ctypes.byref(args), stream_handle(stream)), "decode_layer_step")


def sparse_mla_decode_noalloc(q, kv, slot_idx, scale: float, out, lse, stream=None):
    """echo_sparse_mla_decode without a workspace argument: for callers that may not
    allocate device memory, the library's built-in scratch holds the partials."""
    B, Hq, _ = q.shape
    k = slot_idx.shape[1]
    check(lib().echo_sparse_mla_decode_noalloc(ptr(q), ptr(kv), kv.shape[0], dtype_code(q.dtype), ptr(slot_idx), B,
                                               Hq, k, scale, ptr(out), ptr(lse), stream_handle(stream)),
          "sparse_mla_decode_noalloc")


# ------------------------------------------------------------------- prefill --
def prefill_index(q, w, idx_k, pos0: int, kth_pred, scores, hist, status=None, stream=None):
    """q [Q,64,128] e4m3, w [Q,64] f32, idx_k [Lmax,128] e4m3 -> scores [Q,Lmax], hist [Q,256]."""
    Q, H, D = q.shape
    check(lib().echo_prefill_index(ptr(q), ptr(w), ptr(idx_k), Q, H, D, idx_k.shape[0], pos0, ptr(kth_pred),
                                   ptr(scores), ptr(hist), ptr(status), stream_handle(stream)), "prefill_index")


def prefill_candidates(scores, hist, pos0: int, k: int, kth_pred, bitmap, thr=None, cand_count=None, stream=None):
    Q, Lmax = scores.shape
    check(lib().echo_prefill_candidates(ptr(scores), ptr(hist), Q, Lmax, pos0, k, ptr(kth_pred), ptr(thr),
                                        ptr(cand_count), ptr(bitmap), stream_handle(stream)), "prefill_candidates")


def mark_tokens(tok, bitmap, nbits: int, stream=None):
    rows, row_len = tok.shape
    check(lib().echo_mark_tokens(ptr(tok), rows, row_len, ptr(bitmap), nbits, stream_handle(stream)), "mark_tokens")


def token_list(bitmap, nbits: int, out_list, count, stream=None):
    check(lib().echo_token_list(ptr(bitmap), nbits, ptr(out_list), out_list.numel(), ptr(count),
                                stream_handle(stream)), "token_list")


def translate_slots(layer: LayerCache, tok, host_base, out_slot, stream=None):
    """Slot of every listed token (tok [rows, k], -1 = none); host_base [rows] gives one
    base per row, [1] one base for all rows."""
    rows, k = tok.shape
    per_row = int(host_base.numel() == rows)
    check(lib().echo_translate_slots(layer.ref, ptr(tok), rows, k, ptr(host_base), per_row, ptr(out_slot),
                                     stream_handle(stream)), "translate_slots")


# ------------------------------------------------------------- host pool --
class HostPool:
    """Model-wide host pool: one pinned buffer with every layer's host rows; a request's
    rows are one range shared by all layers (echo_host_pool_*)."""

    def __init__(self, n_layers: int, rows_per_layer: int, kv_dtype=torch.bfloat16, pinned: bool = True):
        code = dtype_code(kv_dtype)
        nbytes = int(lib().echo_host_pool_bytes(n_layers, rows_per_layer, code))
        if nbytes == 0:
            raise EchoError(ERR_INVALID_ARG, "host_pool_bytes")
        self.kv_dtype, self.n_layers, self.rows_per_layer = kv_dtype, int(n_layers), int(rows_per_layer)
        self.buf = torch.empty(n_layers, rows_per_layer, KV_WIDTH, dtype=kv_dtype, pin_memory=pinned)
        self.struct = HostPoolT()
        check(lib().echo_host_pool_init(ctypes.byref(self.struct), self.buf.data_ptr(), n_layers, rows_per_layer,
                                        code), "host_pool_init")

    def alloc(self, rows: int) -> int:
        first = ctypes.c_int64()
        check(lib().echo_host_pool_alloc(ctypes.byref(self.struct), int(rows), ctypes.byref(first)),
              "host_pool_alloc")
        return int(first.value)

    def free(self, first_row: int, rows: int) -> None:
        check(lib().echo_host_pool_free(ctypes.byref(self.struct), int(first_row), int(rows)), "host_pool_free")

    def free_ranges(self) -> list:
        return [(int(self.struct.free_first[i]), int(self.struct.free_rows[i])) for i in range(self.struct.n_free)]

    @property
    def rows_in_use(self) -> int:
        return int(self.struct.rows_in_use)

    def layer_rows(self, layer: int) -> torch.Tensor:
        """Layer `layer`'s rows [rows_per_layer, 576] (a view of the pinned buffer)."""
        host = ctypes.c_void_p()
        check(lib().echo_host_pool_layer(ctypes.byref(self.struct), int(layer), ctypes.byref(host), None),
              "host_pool_layer")
        view = self.buf[layer]
        assert view.data_ptr() == host.value
        return view


# ------------------------------------------------------ block granularity --
def block_scores(scores, seq_len, T: int, bscores, seq_len_blk, stream=None):
    B, Lmax = scores.shape
    check(lib().echo_block_scores(ptr(scores), ptr(seq_len), B, Lmax, int(T), ptr(bscores), ptr(seq_len_blk),
                                  stream_handle(stream)), "block_scores")


def expand_block_slots(sel_blk, block_slot, seq_len, T: int, out, stream=None):
    B, kb = sel_blk.shape
    check(lib().echo_expand_block_slots(ptr(sel_blk), ptr(block_slot), ptr(seq_len), B, kb, int(T), ptr(out),
                                        stream_handle(stream)), "expand_block_slots")
