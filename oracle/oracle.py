"""CPU oracle for the CSA2 attention step (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  The library's product path never touches it.

The arithmetic lives in ``csa2_oracle.c`` (plain loops, double precision);
this module compiles it with gcc, loads it with ctypes and composes the steps
of one CSA2 layer in the order the pages give them:

* Full layer   -- score every visible entry, keep the best 2,048 blocks of 8
  as the candidate pool, take the Top-512 of the pool
  ([P1] "DeepSeek-V4.1-Flash" §3.2; [P2] "DeepSeek-V4.1-Flash 架构详解" §3.2);
* Reindex layer -- rescore only the pool with the layer's own indexer query,
  Top-512 ([P2] §3 mode table, §3.2);
* Reuse layer   -- keep the most recent indices ([P2] §3 mode table);
* every layer   -- attention over the selected entries plus its own FP8
  sliding window under one softmax ([P2] §3, §5 window equation; [P3] §3.3).

Around the layer: the input prologue (RMSNorm of the queries and compressed
KV, then RoPE on their last 64 dims; [P3] §4.3) and the attention options
(sink, output re-rotation, window de-duplication).

Parity status of each function is listed in the design notes; the one
unpinned item is the 890-byte/token decomposition (a footprint reading, not a
function of this module).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_csa2.so")
_lock = threading.Lock()
_lib = None

TOPK = 512
POOL_BLOCKS = 2048
BLOCK = 8
SWA_W = 128


def build(force: bool = False) -> str:
    """Compile the C oracle in place (gcc, OpenMP, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            L.or_e2m1_value.restype = f64
            L.or_e2m1_value.argtypes = [ctypes.c_uint8]
            L.or_e2m1_encode.restype = ctypes.c_uint8
            L.or_e2m1_encode.argtypes = [f64]
            L.or_e4m3_value.restype = f64
            L.or_e4m3_value.argtypes = [ctypes.c_uint8]
            L.or_e4m3_encode.restype = ctypes.c_uint8
            L.or_e4m3_encode.argtypes = [ctypes.c_float]
            L.or_mx_exponent.restype = i32
            L.or_mx_exponent.argtypes = [ctypes.c_float]
            L.or_quant_mxfp4.argtypes = [P, i64, P, P]
            L.or_dequant_mxfp4.argtypes = [P, P, i64, P]
            L.or_quant_fp4_e4m3.argtypes = [P, i64, P, P]
            L.or_dequant_fp4_e4m3.argtypes = [P, P, i64, P]
            L.or_quant_fp8.argtypes = [P, i64, i32, P, P]
            L.or_dequant_fp8.argtypes = [P, P, i64, i32, P]
            L.or_compress.argtypes = [P, P, P, i32, i64, P]
            L.or_index_score.restype = f64
            L.or_index_score.argtypes = [P, P, P, ctypes.c_float]
            L.or_index_scores.argtypes = [P, P, P, P, P, i64, P]
            L.or_topk.restype = i32
            L.or_topk.argtypes = [P, P, i64, i32, P]
            L.or_block_pool.restype = i64
            L.or_block_pool.argtypes = [P, i64, i32, i32, P]
            L.or_attention.argtypes = [P, f64, P, i64, P, f64, i64, P, P]
            L.or_norm_rope.argtypes = [P, i64, i32, P, f64, P, f64, P]
            L.or_num_threads.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(lib().or_num_threads())


# ------------------------------------------------------------------ formats
def e2m1_value(code: int) -> float:
    return lib().or_e2m1_value(code)


def e2m1_encode(v: float) -> int:
    return lib().or_e2m1_encode(v)


def e4m3_value(code: int) -> float:
    return lib().or_e4m3_value(code)


def e4m3_encode(x: float) -> int:
    return lib().or_e4m3_encode(x)


def mx_exponent(amax: float) -> int:
    return lib().or_mx_exponent(amax)


# ------------------------------------------------------------------ compressor, quantisers
def compress(C_bits: np.ndarray, Z_bits: np.ndarray, bias: np.ndarray, m: int) -> np.ndarray:
    """C, Z: [n_tok, 512] bf16 patterns (uint16); bias [m, 512] fp32 -> [n_tok//m, 512] fp32."""
    C = _c(C_bits, np.uint16)
    Z = _c(Z_bits, np.uint16)
    b = _c(bias, np.float32)
    n_tok = C.shape[0]
    out = np.empty((n_tok // m, 512), np.float32)
    lib().or_compress(_p(C), _p(Z), _p(b), m, n_tok, _p(out))
    return out


def quant_mxfp4(x: np.ndarray):
    x = _c(x, np.float32).reshape(-1, 512)
    n = x.shape[0]
    codes = np.empty((n, 256), np.uint8)
    scales = np.empty((n, 16), np.uint8)
    lib().or_quant_mxfp4(_p(x), n, _p(codes), _p(scales))
    return codes, scales


def dequant_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8).reshape(-1, 256)
    scales = _c(scales, np.uint8).reshape(-1, 16)
    out = np.empty((codes.shape[0], 512), np.float64)
    lib().or_dequant_mxfp4(_p(codes), _p(scales), codes.shape[0], _p(out))
    return out


def quant_fp4_e4m3(x: np.ndarray):
    """FP4 entries with one E4M3 scale per 16 elements: codes [n][256], scales [n][32]."""
    x = _c(x, np.float32).reshape(-1, 512)
    n = x.shape[0]
    codes = np.empty((n, 256), np.uint8)
    scales = np.empty((n, 32), np.uint8)
    lib().or_quant_fp4_e4m3(_p(x), n, _p(codes), _p(scales))
    return codes, scales


def dequant_fp4_e4m3(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8).reshape(-1, 256)
    scales = _c(scales, np.uint8).reshape(-1, 32)
    out = np.empty((codes.shape[0], 512), np.float64)
    lib().or_dequant_fp4_e4m3(_p(codes), _p(scales), codes.shape[0], _p(out))
    return out


KV_FORMATS = {0: (quant_mxfp4, dequant_mxfp4, 16), 1: (quant_fp4_e4m3, dequant_fp4_e4m3, 32)}


def quant_fp8(x: np.ndarray):
    x = _c(x, np.float32)
    n, dim = x.shape
    codes = np.empty((n, dim), np.uint8)
    scales = np.empty((n,), np.float32)
    lib().or_quant_fp8(_p(x), n, dim, _p(codes), _p(scales))
    return codes, scales


def dequant_fp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    n, dim = codes.shape
    out = np.empty((n, dim), np.float64)
    lib().or_dequant_fp8(_p(codes), _p(scales), n, dim, _p(out))
    return out


# ------------------------------------------------------------------ indexer score
def index_scores(qi_bits, w, ik_codes, ik_scales, positions=None) -> np.ndarray:
    """Scores (float64) of the entries at ``positions`` (default: all rows)."""
    qi = _c(qi_bits, np.uint16).reshape(32, 128)
    w = _c(w, np.float32).reshape(32)
    codes = _c(ik_codes, np.uint8).reshape(-1, 128)
    sc = _c(ik_scales, np.float32).reshape(-1)
    if positions is None:
        n = codes.shape[0]
        pos_p = None
    else:
        pos = _c(positions, np.int32)
        n = pos.shape[0]
        pos_p = _p(pos)
    out = np.empty((n,), np.float64)
    lib().or_index_scores(_p(qi), _p(w), _p(codes), _p(sc), pos_p, n, _p(out))
    return out


# ------------------------------------------------------------------ selection
def topk(scores: np.ndarray, positions=None, k: int = TOPK) -> np.ndarray:
    """k best (score desc, position asc) positions, returned ascending, -1 padded."""
    s = _c(scores, np.float64)
    n = s.shape[0]
    out = np.empty((k,), np.int32)
    if positions is None:
        lib().or_topk(_p(s), None, n, k, _p(out))
    else:
        pos = _c(positions, np.int32)
        lib().or_topk(_p(s), _p(pos), n, k, _p(out))
    return out


def block_pool(scores: np.ndarray, n_visible: int, blk: int = BLOCK,
               pmax: int = POOL_BLOCKS) -> np.ndarray:
    s = _c(scores[:n_visible], np.float64)
    pool = np.empty((max(pmax * blk, 1),), np.int32)
    npool = lib().or_block_pool(_p(s), n_visible, blk, pmax, _p(pool))
    return pool[:npool].copy()


# ------------------------------------------------------------------ attention
def swa_window(i: int, s: int = 0, W: int = SWA_W):
    """SWAKeys(i) = [max(s, i - W + 1), i] ([P2] §5, bounded-replay window)."""
    return max(int(s), int(i) - W + 1), int(i)


def attention_keys(kv_codes, kv_scales, idx, swa_codes, swa_scales, t: int,
                   swa_start: int = 0, W: int = SWA_W, kv_format: int = 0) -> np.ndarray:
    """Dequantised key set of one query: the selected FP4 entries (idx != -1;
    MXFP4 for kv_format 0, 16-element E4M3-scaled blocks for 1) followed by the
    FP8 window rows of tokens [max(s, t-W+1), t] ([P2] §5 window equation),
    token u held in ring row u % R."""
    sel = np.asarray(idx, np.int64)
    sel = sel[sel >= 0]
    main = KV_FORMATS[kv_format][1](np.asarray(kv_codes)[sel], np.asarray(kv_scales)[sel])
    R = swa_codes.shape[0]
    lo, hi = swa_window(t, swa_start, W)
    toks = np.arange(lo, hi + 1, dtype=np.int64)
    rows = toks % R
    swa = dequant_fp8(np.asarray(swa_codes)[rows].reshape(-1, 512),
                      np.asarray(swa_scales)[rows].reshape(-1))
    return np.concatenate([main, swa], axis=0)


def attention(q_bits, sm_scale: float, keys: np.ndarray, sink=None, rope_base: float = 0.0, t: int = 0):
    """o [64, 512] fp32, lse [64] fp32 of one query over dequantised keys.
    sink: optional per-head logits joining the softmax denominator; rope_base > 0:
    the output's RoPE dims rotated back by the query position t (see the C source)."""
    q = _c(q_bits, np.uint16).reshape(64, 512)
    k = _c(keys, np.float64).reshape(-1, 512)
    z = None if sink is None else _c(sink, np.float64).reshape(64)
    o = np.empty((64, 512), np.float32)
    lse = np.empty((64,), np.float32)
    lib().or_attention(_p(q), float(sm_scale), _p(k), k.shape[0], None if z is None else _p(z), float(rope_base),
                       int(t), _p(o), _p(lse))
    return o, lse


def norm_rope(x, gamma=None, eps: float = 1e-6, pos=None, rope_base: float = 0.0) -> np.ndarray:
    """float64 [rows][vecs][512]: RMSNorm of every 512-dim vector, then the
    forward RoPE of its last 64 dims at the row's position (see the C source)."""
    xx = _c(x, np.float64)
    assert xx.ndim == 3 and xx.shape[2] == 512
    rows, vecs = xx.shape[0], xx.shape[1]
    g = None if gamma is None else _c(gamma, np.float64).reshape(512)
    p = np.zeros((max(rows, 1),), np.int64) if pos is None else _c(pos, np.int64).reshape(rows)
    out = np.empty_like(xx)
    lib().or_norm_rope(_p(xx), rows * vecs, max(vecs, 1), None if g is None else _p(g), float(eps), _p(p),
                       float(rope_base), _p(out))
    return out


def dedup_selection(positions, t: int, m: int, swa_start: int = 0, W: int = SWA_W) -> np.ndarray:
    """The selected positions without those whose token is also a window row
    (m = 1 only: a compressed entry of m > 1 tokens is not a window row)."""
    pos = np.asarray(positions, np.int64)
    if m != 1:
        return pos
    lo, hi = swa_window(t, swa_start, W)
    return pos[(pos < lo) | (pos > hi)]


# ------------------------------------------------------------------ layers
def n_visible(t: int, m: int, n_entries: int) -> int:
    """Entries visible to the query at token t: entry j covers tokens
    [j*m, j*m+m) and is visible once complete, (j+1)*m - 1 <= t ([P3] §3.3:
    a query cannot see the rest of its own unfinished compression block)."""
    return max(0, min(n_entries, (t + 1) // m))


def full_select(qi_bits, w, ik_codes, ik_scales, nvis: int):
    """Full layer: score all visible entries, block pool, Top-512 of the pool.
    Returns (idx, pool, scores)."""
    scores = index_scores(qi_bits, w, ik_codes[:nvis], ik_scales[:nvis])
    pool = block_pool(scores, nvis)
    idx = topk(scores[pool], pool)
    return idx, pool, scores


def reindex_select(qi_bits, w, ik_codes, ik_scales, pool):
    """Reindex layer: rescore the pool positions only, Top-512.  Returns (idx, pool_scores)."""
    ps = index_scores(qi_bits, w, ik_codes, ik_scales, positions=pool)
    return topk(ps, pool), ps


DECODER_PATTERN = ["full", "reuse", "reuse", "reuse"] + ["reindex", "reuse", "reuse", "reuse"] * 4
ENCODER_GROUP = ["full"] + ["reuse"] * 5
