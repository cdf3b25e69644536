"""Python binding of the CSA2 C ABI (include/csa2.h).

Argument marshalling only: every function here checks dtypes / devices of
torch tensors, turns them into raw device pointers and calls the entry point
of the same name in ``libcsa2.so`` on the current torch CUDA stream.  There is
no fallback: if the library is missing or a call fails, a Python exception is
raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

HEADS, HEAD_DIM, IDX_HEADS, IDX_DIM = 64, 512, 32, 128
TOPK, BLOCK, POOL_BLOCKS, POOL_MAX, SWA_WINDOW, PAGE = 512, 8, 2048, 16384, 128, 64
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
KV_MXFP4, KV_FP4_E4M3 = 0, 1                  # main-KV formats: scale bytes per entry 16 / 32
KV_SCALE_BYTES = {KV_MXFP4: 16, KV_FP4_E4M3: 32}
MODES = {"full": MODE_FULL, "reindex": MODE_REINDEX, "reuse": MODE_REUSE}
DEV_BAD_PAGE, DEV_BAD_SLOT, DEV_TIMEOUT, DEV_BAD_INDEX = 1, 2, 4, 8

_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class Cache(ctypes.Structure):
    _fields_ = [("kv_codes", _vp), ("kv_scales", _vp), ("ik_codes", _vp), ("ik_scales", _vp),
                ("num_slots", _i64), ("block_table", _vp), ("max_pages", _i32), ("kv_format", _i32),
                ("status", _vp)]


class Batch(ctypes.Structure):
    _fields_ = [("batch", _i32), ("nq", _i32), ("m", _i32), ("pad_", _i32), ("max_entries", _i64),
                ("n_entries", _vp), ("q_pos", _vp)]


class Swa(ctypes.Structure):
    _fields_ = [("codes", _vp), ("scales", _vp), ("rows", _i32), ("flags", _i32), ("start", _vp), ("new_rows", _vp),
                ("sink", _vp), ("rope_base", _f32), ("pad_", _i32)]


class LayerIO(ctypes.Structure):
    _fields_ = [("q", _vp), ("qi", _vp), ("w", _vp), ("swa", Swa), ("sm_scale", _f32), ("flags", _i32),
                ("idx", _vp), ("pool", _vp), ("pool_len", _vp), ("o", _vp), ("lse", _vp),
                ("prof_begin", _vp), ("prof_end", _vp)]


EXPORTS = {
    "csa2_compress": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i64, _vp, _vp]),
    "csa2_quant_mxfp4": (ctypes.c_int, [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _vp]),
    "csa2_quant_fp8": (ctypes.c_int, [_vp, _i64, _i32, _vp, _vp, _vp, _i64, _vp, _vp]),
    "csa2_quant_fp4_e4m3": (ctypes.c_int, [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _vp]),
    "csa2_append_entries": (ctypes.c_int, [ctypes.POINTER(Cache), _vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp]),
    "csa2_norm_rope": (ctypes.c_int, [_vp, _i64, _i32, _vp, _f32, _vp, _f32, _vp, _vp, _vp]),
    "csa2_index_scores": (ctypes.c_int, [ctypes.POINTER(Cache), ctypes.POINTER(Batch), _vp, _vp, _vp, _vp,
                                         _vp, _i64, _vp]),
    "csa2_index_scores_pool": (ctypes.c_int, [ctypes.POINTER(Cache), ctypes.POINTER(Batch), _vp, _vp, _vp,
                                              _vp, _i64, _vp, _vp, _sz, _vp]),
    "csa2_index_scores_pool_workspace_size": (_sz, [ctypes.POINTER(Batch), _i64]),
    "csa2_topk": (ctypes.c_int, [_vp, _i64, _vp, _i32, _vp, _i32, _vp, _vp]),
    "csa2_topk_blocks": (ctypes.c_int, [_vp, _i64, _vp, _i32, _i32, _vp, _vp, _vp]),
    "csa2_sparse_attn": (ctypes.c_int, [ctypes.POINTER(Cache), ctypes.POINTER(Batch), _vp, _f32, _vp, _i32,
                                        ctypes.POINTER(Swa), _vp, _vp, _vp, _sz, _vp]),
    "csa2_sparse_attn_workspace_size": (_sz, [_i32, _i32]),
    "csa2_sparse_attn_schedule": (ctypes.c_int, [ctypes.POINTER(Batch), ctypes.POINTER(Swa)]),
    "csa2_layer": (ctypes.c_int, [_i32, ctypes.POINTER(Cache), ctypes.POINTER(Batch), ctypes.POINTER(LayerIO),
                                  _vp, _sz, _vp]),
    "csa2_layer_workspace_size": (_sz, [_i32, ctypes.POINTER(Batch)]),
    "csa2_layer_noalloc": (ctypes.c_int, [_i32, ctypes.POINTER(Cache), ctypes.POINTER(Batch),
                                          ctypes.POINTER(LayerIO), _vp]),
    "csa2_debug_set_wait_limit": (ctypes.c_int, [ctypes.c_uint32]),
    "csa2_status_string": (ctypes.c_char_p, [_i32]),
    "csa2_last_cuda_error": (_i32, []),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libcsa2.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"CSA2 CUDA library not built: {path} is missing "
                              "(run compressed_sparse_attention_layer_gb300.build.build())")
        lib = ctypes.CDLL(path)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class Csa2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = load()
        msg = lib.csa2_status_string(status).decode()
        if status == -7:
            msg += f" (cudaError {lib.csa2_last_cuda_error()})"
        super().__init__(f"{fn}: status {status}: {msg}")
        self.status = status


def _check(fn: str, status: int):
    if status != 0:
        raise Csa2Error(fn, status)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------- descriptors
class PagedCache:
    """Device buffers of the layer-shared cache (caller-side allocation)."""

    def __init__(self, num_pages: int, block_table: torch.Tensor, device="cuda", kv_format: int = KV_MXFP4):
        self.num_pages = int(num_pages)
        self.kv_format = int(kv_format)
        S = self.num_pages * PAGE
        self.kv_codes = torch.zeros((S, 256), dtype=torch.uint8, device=device)
        self.kv_scales = torch.zeros((S, KV_SCALE_BYTES[self.kv_format]), dtype=torch.uint8, device=device)
        self.ik_codes = torch.zeros((S, 128), dtype=torch.uint8, device=device)
        self.ik_scales = torch.ones((S,), dtype=torch.float32, device=device)
        self.block_table = block_table.to(device=device, dtype=torch.int32).contiguous()
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)

    @property
    def num_slots(self):
        return self.num_pages * PAGE

    def struct(self) -> Cache:
        return Cache(_ptr(self.kv_codes), _ptr(self.kv_scales), _ptr(self.ik_codes), _ptr(self.ik_scales),
                     self.num_slots, _ptr(self.block_table, torch.int32), self.block_table.shape[1],
                     self.kv_format, _ptr(self.status))

    def slots(self, b: int, entries: torch.Tensor) -> torch.Tensor:
        """Slot ids of logical entries of sequence b (a host-side helper for appends)."""
        e = entries.to(torch.int64)
        return self.block_table[b].to(torch.int64)[e // PAGE] * PAGE + e % PAGE


def batch_struct(n_entries: torch.Tensor, q_pos: torch.Tensor, nq: int, m: int, max_entries: int) -> Batch:
    return Batch(n_entries.shape[0], nq, m, 0, int(max_entries), _ptr(n_entries, torch.int64, "n_entries"),
                 _ptr(q_pos, torch.int64, "q_pos"))


ATTN_DEDUP_WINDOW = 1
LAYER_SCORES_BF16 = 1      # csa2_layer_io.flags: selection on bf16-rounded index scores
LAYER_INDEX_E4M3_QUERY = 2  # csa2_layer_io.flags: the Full scan's query as one e4m3 part per head
ATTN_EARLY_INPUTS = 2      # REUSE layers: keys loaded while the previous layer finishes (see the header)
ATTN_EARLY_ALL = 16        # REUSE layers: the whole attention before the dependency wait (see the header)
ATTN_SCHEDULE_CHUNKS = 4   # attention: one cluster per (row, key chunk) and a merge kernel
ATTN_SCHEDULE_ROWS = 8     # attention: persistent clusters over whole rows (many rows; no new_rows)


def swa_struct(codes: torch.Tensor, scales: torch.Tensor, start=None, new_rows=None, sink=None,
               rope_base: float = 0.0, flags: int = 0) -> Swa:
    """new_rows: optional fp32 [B][512] window rows of the decode tokens, quantised
    into the ring by the attention call itself; sink: optional fp32 [64] per-head
    sink logits; rope_base > 0 rotates the output's RoPE dims back by the query
    position; flags: ATTN_DEDUP_WINDOW | ATTN_EARLY_INPUTS | ATTN_EARLY_ALL |
    ATTN_SCHEDULE_CHUNKS or ATTN_SCHEDULE_ROWS."""
    return Swa(_ptr(codes, torch.uint8, "swa codes"), _ptr(scales, torch.float32, "swa scales"), codes.shape[1],
               int(flags), _ptr(start, torch.int64, "swa start"), _ptr(new_rows, torch.float32, "swa new rows"),
               _ptr(sink, torch.float32, "sink"), float(rope_base), 0)


# ---------------------------------------------------------------- entry points
def csa2_compress(C, Z, bias, m: int, out, stream=None):
    _check("csa2_compress", load().csa2_compress(_ptr(C, torch.bfloat16, "C"), _ptr(Z, torch.bfloat16, "Z"),
                                                 _ptr(bias, torch.float32, "bias"), m, C.shape[0],
                                                 _ptr(out, torch.float32, "out"), _stream(stream)))


def csa2_quant_mxfp4(x, codes, scales, slots=None, status=None, stream=None):
    _check("csa2_quant_mxfp4", load().csa2_quant_mxfp4(
        _ptr(x, torch.float32, "x"), x.shape[0], _ptr(slots, torch.int64, "slots"), _ptr(codes, torch.uint8),
        _ptr(scales, torch.uint8), codes.shape[0], _ptr(status, torch.int32), _stream(stream)))


def csa2_quant_fp4_e4m3(x, codes, scales, slots=None, status=None, stream=None):
    """FP4 with one E4M3 scale per 16 elements: codes [S][256], scales [S][32]."""
    _check("csa2_quant_fp4_e4m3", load().csa2_quant_fp4_e4m3(
        _ptr(x, torch.float32, "x"), x.shape[0], _ptr(slots, torch.int64, "slots"), _ptr(codes, torch.uint8),
        _ptr(scales, torch.uint8), codes.shape[0], _ptr(status, torch.int32), _stream(stream)))


def csa2_quant_fp8(x, codes, scales, slots=None, status=None, stream=None):
    _check("csa2_quant_fp8", load().csa2_quant_fp8(
        _ptr(x, torch.float32, "x"), x.shape[0], x.shape[1], _ptr(slots, torch.int64, "slots"),
        _ptr(codes, torch.uint8), _ptr(scales, torch.float32), codes.shape[0], _ptr(status, torch.int32),
        _stream(stream)))


def csa2_append_entries(cache, C, Z, bias, m: int, ik, slots=None, entries=None, stream=None):
    """A step's new entries: compress C/Z (bf16 [n_tok][512]) into n_tok // m
    entries, quantise them into cache's main KV and ik (fp32 [n_ent][128])
    into its indexer keys, at slots (int64 [n_ent]); entries: optional fp32
    [n_ent][512] copy of the compressed entries.  cache: a csa2.Cache struct."""
    _check("csa2_append_entries", load().csa2_append_entries(
        ctypes.byref(cache), _ptr(C, torch.bfloat16, "C"), _ptr(Z, torch.bfloat16, "Z"),
        _ptr(bias, torch.float32, "bias"), m, C.shape[0], _ptr(ik, torch.float32, "ik"),
        _ptr(slots, torch.int64, "slots"), _ptr(entries, torch.float32, "entries"), _stream(stream)))


def csa2_norm_rope(x, out, gamma=None, eps: float = 1e-6, pos=None, rope_base: float = 0.0, stream=None):
    """RMSNorm and forward partial RoPE of x fp32 [rows][vecs][512] into out
    (fp32 or bf16, same shape; out may be x when fp32); pos int64 [rows]."""
    assert x.dim() == 3 and x.shape[2] == 512 and tuple(out.shape) == tuple(x.shape)
    f32 = out.dtype == torch.float32
    _check("csa2_norm_rope", load().csa2_norm_rope(
        _ptr(x, torch.float32, "x"), x.shape[0], x.shape[1], _ptr(gamma, torch.float32, "gamma"), float(eps),
        _ptr(pos, torch.int64, "pos"), float(rope_base), _ptr(out, torch.float32, "out") if f32 else None,
        None if f32 else _ptr(out, torch.bfloat16, "out"), _stream(stream)))


def csa2_index_scores(cache: Cache, batch: Batch, qi, w, scores=None, block_max=None, n_visible=None,
                      ld: int = None, stream=None):
    _check("csa2_index_scores", load().csa2_index_scores(
        ctypes.byref(cache), ctypes.byref(batch), _ptr(qi, torch.bfloat16, "qi"), _ptr(w, torch.float32, "w"),
        _ptr(scores, torch.float32), _ptr(block_max, torch.float32), _ptr(n_visible, torch.int32), ld,
        _stream(stream)))


def csa2_index_scores_pool_workspace_size(batch: Batch, ld: int) -> int:
    return int(load().csa2_index_scores_pool_workspace_size(ctypes.byref(batch), int(ld)))


def csa2_index_scores_pool(cache: Cache, batch: Batch, qi, w, pool, pool_len, scores, workspace=None, stream=None):
    """workspace: uint8 device buffer of csa2_index_scores_pool_workspace_size bytes (allocated
    here through torch when None)."""
    ld = pool.shape[-1]
    if workspace is None:
        workspace = torch.empty(csa2_index_scores_pool_workspace_size(batch, ld), dtype=torch.uint8,
                                device=pool.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("csa2_index_scores_pool", load().csa2_index_scores_pool(
        ctypes.byref(cache), ctypes.byref(batch), _ptr(qi, torch.bfloat16, "qi"), _ptr(w, torch.float32, "w"),
        _ptr(pool, torch.int32, "pool"), _ptr(pool_len, torch.int32, "pool_len"), ld,
        _ptr(scores, torch.float32, "scores"), _ptr(workspace), ws_bytes, _stream(stream)))


def csa2_topk(scores, lens, k: int, out, cand=None, stream=None):
    rows = lens.shape[0]
    _check("csa2_topk", load().csa2_topk(_ptr(scores, torch.float32, "scores"), scores.shape[-1],
                                         _ptr(lens, torch.int32, "len"), rows, _ptr(cand, torch.int32, "cand"),
                                         k, _ptr(out, torch.int32, "out"), _stream(stream)))


def csa2_topk_blocks(block_max, n_visible, pmax: int, pool, pool_len, stream=None):
    rows = n_visible.shape[0]
    _check("csa2_topk_blocks", load().csa2_topk_blocks(
        _ptr(block_max, torch.float32, "block_max"), block_max.shape[-1], _ptr(n_visible, torch.int32),
        rows, pmax, _ptr(pool, torch.int32, "pool"), _ptr(pool_len, torch.int32, "pool_len"), _stream(stream)))


def csa2_sparse_attn_workspace_size(batch: int, nq: int) -> int:
    return int(load().csa2_sparse_attn_workspace_size(batch, nq))


def csa2_sparse_attn_schedule(batch: Batch, swa: Swa) -> int:
    """ATTN_SCHEDULE_CHUNKS or ATTN_SCHEDULE_ROWS: the schedule the attention takes."""
    r = int(load().csa2_sparse_attn_schedule(ctypes.byref(batch), ctypes.byref(swa)))
    _check("csa2_sparse_attn_schedule", min(r, 0))
    return r


def csa2_sparse_attn(cache: Cache, batch: Batch, q, sm_scale: float, idx, swa: Swa, o, lse, workspace=None,
                     stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("csa2_sparse_attn", load().csa2_sparse_attn(
        ctypes.byref(cache), ctypes.byref(batch), _ptr(q, torch.bfloat16, "q"), float(sm_scale),
        _ptr(idx, torch.int32, "idx"), idx.shape[-1], ctypes.byref(swa), _ptr(o, torch.float32, "o"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace), ws_bytes, _stream(stream)))


def csa2_layer_workspace_size(mode: int, batch: Batch) -> int:
    return int(load().csa2_layer_workspace_size(mode, ctypes.byref(batch)))


def layer_io(q, qi, w, swa: Swa, sm_scale, idx, pool, pool_len, o, lse, prof=None, flags: int = 0) -> LayerIO:
    """prof: optional (begin, end) pair of recorded torch.cuda.Event(enable_timing=True).
    flags: LAYER_SCORES_BF16 | LAYER_INDEX_E4M3_QUERY or 0."""
    pb, pe = (prof[0].cuda_event, prof[1].cuda_event) if prof else (None, None)
    return LayerIO(_ptr(q, torch.bfloat16, "q"), _ptr(qi, torch.bfloat16, "qi"), _ptr(w, torch.float32, "w"),
                   swa, float(sm_scale), int(flags), _ptr(idx, torch.int32, "idx"), _ptr(pool, torch.int32, "pool"),
                   _ptr(pool_len, torch.int32, "pool_len"), _ptr(o, torch.float32, "o"),
                   _ptr(lse, torch.float32, "lse"), pb, pe)


def csa2_layer(mode: int, cache: Cache, batch: Batch, io: LayerIO, workspace, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("csa2_layer", load().csa2_layer(int(mode), ctypes.byref(cache), ctypes.byref(batch), ctypes.byref(io),
                                           _ptr(workspace), ws_bytes, _stream(stream)))


def csa2_layer_noalloc(mode: int, cache: Cache, batch: Batch, io: LayerIO, stream=None):
    """csa2_layer with the library's static scratch instead of a caller workspace."""
    _check("csa2_layer_noalloc", load().csa2_layer_noalloc(int(mode), ctypes.byref(cache), ctypes.byref(batch),
                                                           ctypes.byref(io), _stream(stream)))


def csa2_debug_set_wait_limit(polls: int):
    """Polls after which a bounded device wait gives up, for launches after the call
    (0: the default).  A test hook for the timeout path."""
    _check("csa2_debug_set_wait_limit", load().csa2_debug_set_wait_limit(int(polls)))
