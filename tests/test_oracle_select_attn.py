"""Pins of the oracle's selection (Full, Reindex and Reuse layers) and attention.

Anchors: numpy's lexsort (an independent sort) for Top-K order and ties, a
brute-force block pool, the pool-versus-global equivalence that holds for
max-aggregated blocks, torch's scaled_dot_product_attention in float64 for
the softmax, and closed forms (one key, identical keys, no keys).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_layer_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _lexsort_topk(scores, positions, k):
    order = np.lexsort((positions, -scores))        # score desc, position asc
    chosen = np.sort(positions[order[:k]])
    out = np.full(k, -1, np.int32)
    out[:chosen.size] = chosen
    return out


# ---------------------------------------------------------------- Top-K
@pytest.mark.parametrize("n", [0, 1, 7, 511, 512, 513, 5000])
def test_topk_matches_lexsort(n):
    rng = np.random.default_rng(n)
    s = rng.integers(0, 50, n).astype(np.float64)     # many ties
    pos = np.arange(n, dtype=np.int32)
    assert np.array_equal(oracle.topk(s), _lexsort_topk(s, pos, 512))
    # scattered candidate positions
    cand = np.sort(rng.choice(10 * n + 1, n, replace=False)).astype(np.int32)
    assert np.array_equal(oracle.topk(s, cand), _lexsort_topk(s, cand, 512))


def test_topk_all_equal_takes_lowest_positions():
    s = np.full(3000, 2.5)
    assert np.array_equal(oracle.topk(s), np.arange(512))


def test_block_pool_brute_force():
    rng = np.random.default_rng(3)
    for n in [1, 8, 9, 100, 16383, 16384, 16385, 40000]:
        s = rng.integers(0, 1000, n).astype(np.float64)
        pool = oracle.block_pool(s, n)
        nb = (n + 7) // 8
        pad = np.full(nb * 8, -np.inf)
        pad[:n] = s
        bmax = pad.reshape(nb, 8).max(axis=1)
        keep = np.sort(np.lexsort((np.arange(nb), -bmax))[:2048])
        want = np.concatenate([np.arange(b * 8, min(b * 8 + 8, n)) for b in keep])
        assert np.array_equal(pool, want)
        assert pool.size <= 16384


def test_pool_top512_equals_global_top512():
    # every global top-512 position sits in a block whose max is at least the
    # 512th score, so at most 512 such blocks, all ranked inside the top 2,048
    rng = np.random.default_rng(4)
    for n in [20000, 100000]:
        s = rng.standard_normal(n) ** 2
        s[rng.integers(0, n, 300)] = 3.0             # ties across blocks
        pool = oracle.block_pool(s, n)
        assert np.array_equal(oracle.topk(s[pool], pool), oracle.topk(s))


# ---------------------------------------------------------------- attention
def _q(seed):
    return synth.normal_bf16(synth.stream_id(seed, 1), 0, 64 * 512, sigma=512 ** -0.5).reshape(64, 512)


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(9)
    qb = _q(9)
    keys = oracle.dequant_mxfp4(*oracle.quant_mxfp4(rng.standard_normal((300, 512)).astype(np.float32)))
    for scale in (1.0, 0.5):
        o, lse = oracle.attention(qb, scale, keys)
        q = torch.from_numpy(synth.bf16_bits_to_f32(qb).astype(np.float64))
        k = torch.from_numpy(keys)
        ref = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], k[None], scale=scale)[0]
        ref_lse = torch.logsumexp(scale * q @ k.T, dim=1)
        assert np.allclose(o, ref.numpy(), rtol=1e-6, atol=1e-7)
        assert np.allclose(lse, ref_lse.numpy(), rtol=1e-6, atol=1e-6)


def test_attention_closed_forms():
    qb = _q(10)
    rng = np.random.default_rng(10)
    k1 = oracle.dequant_fp8(*oracle.quant_fp8(rng.standard_normal((1, 512)).astype(np.float32)))
    o, lse = oracle.attention(qb, 1.0, k1)
    assert np.array_equal(o, np.broadcast_to(k1.astype(np.float32), (64, 512)))      # one key: o = k
    q = synth.bf16_bits_to_f32(qb).astype(np.float64)
    assert np.allclose(lse, q @ k1[0], rtol=1e-6, atol=1e-7)          # lse is stored in fp32
    o, lse = oracle.attention(qb, 1.0, np.repeat(k1, 37, axis=0))                    # identical keys
    assert np.array_equal(o, np.broadcast_to(k1.astype(np.float32), (64, 512)))
    assert np.allclose(lse, q @ k1[0] + np.log(37.0), rtol=1e-6, atol=1e-6)
    o, lse = oracle.attention(qb, 1.0, np.zeros((0, 512)))                           # no keys
    assert not o.any() and np.all(np.isneginf(lse))


def test_attention_key_order_invariant():
    qb = _q(11)
    rng = np.random.default_rng(11)
    keys = rng.standard_normal((200, 512))
    o, lse = oracle.attention(qb, 1.0, keys)
    p = rng.permutation(200)
    o2, lse2 = oracle.attention(qb, 1.0, keys[p])
    assert np.allclose(o, o2, rtol=1e-6, atol=1e-7) and np.allclose(lse, lse2, rtol=1e-7)


def test_swa_window_fixture():
    with open(os.path.join(GOLD, "swa_window.txt")) as f:
        rows = [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]
    for i, s, W, lo, hi in rows:
        assert oracle.swa_window(i, s, W) == (lo, hi)


def test_attention_keys_selection_and_window():
    rng = np.random.default_rng(12)
    E = 64
    kvc, kvs = oracle.quant_mxfp4(rng.standard_normal((E, 512)).astype(np.float32))
    R = 128
    swc, sws = oracle.quant_fp8(rng.standard_normal((R, 512)).astype(np.float32))
    idx = np.array([3, 10, -1, -1], np.int32)
    t = 300                                  # window tokens 173..300 in ring rows t % 128
    keys = oracle.attention_keys(kvc, kvs, idx, swc, sws, t)
    assert keys.shape == (2 + 128, 512)
    assert np.array_equal(keys[0], oracle.dequant_mxfp4(kvc[3:4], kvs[3:4])[0])
    assert np.array_equal(keys[2], oracle.dequant_fp8(swc[173 % R:173 % R + 1], sws[173 % R:173 % R + 1])[0])
    keys = oracle.attention_keys(kvc, kvs, idx, swc, sws, 5)          # young sequence: 6 window rows
    assert keys.shape == (2 + 6, 512)
    keys = oracle.attention_keys(kvc, kvs, idx, swc, sws, 300, swa_start=290)   # replay start
    assert keys.shape == (2 + 11, 512)


# ---------------------------------------------------------------- layers
def _small_problem(N, seed, planted_blocks=()):
    ik_src = synth.normal_f32(synth.stream_id(seed, 2), 0, N * 128).reshape(N, 128)
    qi = synth.normal_bf16(synth.stream_id(seed, 3), 0, 4096).reshape(32, 128)
    w = synth.uniform_f32(synth.stream_id(seed, 4), 0, 32)
    if planted_blocks:
        u = (w.astype(np.float64)[:, None] * synth.bf16_bits_to_f32(qi).astype(np.float64)).sum(0)
        u /= np.linalg.norm(u)
        for b in planted_blocks:
            ik_src[b * 8:(b + 1) * 8] = (np.linalg.norm(ik_src[b * 8:(b + 1) * 8], axis=1)[:, None] * 0.9 * u).astype(np.float32)
    codes, scales = oracle.quant_fp8(ik_src)
    return qi, w, codes, scales


def test_full_layer_small_context_is_plain_topk():
    # 4,096 entries = 512 blocks <= 2,048: the pool is every position, so the
    # hierarchy reduces to one Top-512 over all scores
    qi, w, codes, scales = _small_problem(4096, 31)
    idx, pool, scores = oracle.full_select(qi, w, codes, scales, 4096)
    assert np.array_equal(pool, np.arange(4096))
    assert np.array_equal(idx, _lexsort_topk(scores, np.arange(4096, dtype=np.int32), 512))


def test_reindex_with_full_query_reproduces_full():
    qi, w, codes, scales = _small_problem(30000, 32)
    idx, pool, scores = oracle.full_select(qi, w, codes, scales, 30000)
    assert pool.size == 16384
    idx2, _ = oracle.reindex_select(qi, w, codes, scales, pool)
    assert np.array_equal(idx, idx2)


def test_planted_blocks_recovered():
    planted = [5, 100, 777, 2000, 3333]
    qi, w, codes, scales = _small_problem(30000, 33, planted)
    idx, pool, _ = oracle.full_select(qi, w, codes, scales, 30000)
    want = np.concatenate([np.arange(b * 8, b * 8 + 8) for b in planted])
    assert np.isin(want, idx).all()
    assert np.isin(want, pool).all()


def test_dense_cross_check_when_topk_covers_context():
    # N <= 512 entries: Top-512 selects every visible entry, so sparse attention
    # equals dense attention over all entries plus the window
    rng = np.random.default_rng(40)
    for N in [1, 7, 64, 512]:
        qi, w, codes, scales = _small_problem(N, 40 + N)
        idx, pool, _ = oracle.full_select(qi, w, codes, scales, N)
        assert np.array_equal(np.sort(idx[idx >= 0]), np.arange(N))
        kvc, kvs = oracle.quant_mxfp4(rng.standard_normal((N, 512)).astype(np.float32))
        swc, sws = oracle.quant_fp8(rng.standard_normal((128, 512)).astype(np.float32))
        qb = _q(40 + N)
        t = N - 1
        o, lse = oracle.attention(qb, 1.0, oracle.attention_keys(kvc, kvs, idx, swc, sws, t))
        rows = np.arange(max(0, t - 127), t + 1) % 128
        dense = np.concatenate([oracle.dequant_mxfp4(kvc, kvs), oracle.dequant_fp8(swc[rows], sws[rows])])
        q = torch.from_numpy(synth.bf16_bits_to_f32(qb).astype(np.float64))
        k = torch.from_numpy(dense)
        ref = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], k[None], scale=1.0)[0]
        assert np.allclose(o, ref.numpy(), rtol=1e-6, atol=1e-7)


def test_visibility_rule():
    # entry j (tokens jm..jm+m-1) becomes visible at token (j+1)m-1
    assert oracle.n_visible(0, 2, 100) == 0
    assert oracle.n_visible(1, 2, 100) == 1
    assert oracle.n_visible(2, 2, 100) == 1
    assert oracle.n_visible(73727, 2, 36864) == 36864
    assert oracle.n_visible(65536, 2, 36864) == 32768
    assert oracle.n_visible(1048575, 1, 1048576) == 1048576


# ---------------------------------------------------------------- attention options
# [P3] §4.3 names a learnable attention sink and partial RoPE on the last 64
# dims with the output rotated back; the window de-duplication is the option
# of reading c12 (one softmax over both key sets by default).
def _q_and_keys(seed, nk):
    rng = np.random.default_rng(seed)
    qb = torch.from_numpy((rng.standard_normal((64, 512)) / np.sqrt(512)).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    keys = rng.standard_normal((nk, 512))
    return qb, keys


def test_sink_minus_inf_is_no_sink():
    qb, keys = _q_and_keys(31, 40)
    o, lse = oracle.attention(qb, 1.0, keys)
    o2, lse2 = oracle.attention(qb, 1.0, keys, sink=np.full(64, -np.inf))
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_sink_closed_forms():
    qb, keys = _q_and_keys(32, 1)
    q = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).double().numpy()
    z = np.linspace(-3, 3, 64)
    o, lse = oracle.attention(qb, 1.0, keys, sink=z)
    l = q @ keys[0]                                   # one key: o_h = k sigma(l_h - z_h)
    w = 1.0 / (1.0 + np.exp(z - l))
    assert np.allclose(o, w[:, None] * keys[0][None, :], rtol=1e-6, atol=1e-7)
    assert np.allclose(lse, np.logaddexp(l, z), rtol=1e-6, atol=1e-6)
    # many keys: lse with a sink = logaddexp(lse without it, z); o scales by the kept mass
    qb, keys = _q_and_keys(33, 70)
    o0, lse0 = oracle.attention(qb, 1.0, keys)
    o1, lse1 = oracle.attention(qb, 1.0, keys, sink=z)
    assert np.allclose(lse1, np.logaddexp(lse0.astype(np.float64), z), rtol=1e-6, atol=1e-6)
    kept = np.exp(lse0.astype(np.float64) - np.logaddexp(lse0.astype(np.float64), z))
    assert np.allclose(o1, o0 * kept[:, None], rtol=1e-5, atol=1e-7)
    # no keys, a finite sink: o = 0, lse = z
    o, lse = oracle.attention(qb, 1.0, np.zeros((0, 512)), sink=z)
    assert np.all(o == 0) and np.allclose(lse, z.astype(np.float32))


def test_output_rerotation():
    qb, keys = _q_and_keys(34, 50)
    o0, lse0 = oracle.attention(qb, 1.0, keys)
    same, _ = oracle.attention(qb, 1.0, keys, rope_base=10000.0, t=0)
    assert np.array_equal(same, o0)                                     # t = 0: identity
    t = 987654
    o1, lse1 = oracle.attention(qb, 1.0, keys, rope_base=10000.0, t=t)
    assert np.array_equal(lse1, lse0)
    assert np.array_equal(o1[:, :448], o0[:, :448])                     # only the last 64 dims move
    # independent check: pairs (448+i, 480+i) as complex numbers times e^{-i t w_i}
    w = 10000.0 ** (-np.arange(32) / 32.0)
    zc = (o0[:, 448:480].astype(np.float64) + 1j * o0[:, 480:512]) * np.exp(-1j * np.mod(t * w, 2 * np.pi))
    assert np.allclose(o1[:, 448:480], zc.real, atol=2e-7)
    assert np.allclose(o1[:, 480:512], zc.imag, atol=2e-7)


def test_dedup_selection():
    t = 1000
    sel = np.array([5, 871, 872, 873, 900, 999, 1000], np.int64)        # window of t: [873, 1000]
    assert np.array_equal(oracle.dedup_selection(sel, t, 1), [5, 871, 872])
    assert np.array_equal(oracle.dedup_selection(sel, t, 2), sel)      # compressed entries stay
    assert np.array_equal(oracle.dedup_selection(sel, 50, 1), sel[sel > 50])
    assert np.array_equal(oracle.dedup_selection(sel, t, 1, swa_start=950), [5, 871, 872, 873, 900])


# ---------------------------------------------------------------- norm / RoPE prologue
def test_norm_rope_closed_forms():
    # a constant vector c: mean square c^2, y = c / sqrt(c^2 + eps) * gamma
    x = np.full((2, 3, 512), -2.0)
    assert np.allclose(oracle.norm_rope(x, eps=0.0), -1.0, rtol=0, atol=1e-15)
    assert np.allclose(oracle.norm_rope(x, eps=1.0), -2.0 / np.sqrt(5.0), rtol=0, atol=1e-15)
    g = np.linspace(0.5, 1.5, 512)
    assert np.allclose(oracle.norm_rope(x, gamma=g, eps=0.0)[1, 2], -g, rtol=0, atol=1e-15)
    # a one-hot vector e_d * s: mean square s^2 / 512, so y_d = sqrt(512) (eps = 0)
    x = np.zeros((1, 1, 512))
    x[0, 0, 17] = 0.25
    y = oracle.norm_rope(x, eps=0.0)
    assert abs(y[0, 0, 17] - np.sqrt(512.0)) < 1e-12 and np.count_nonzero(y) == 1
    # a zero vector with eps > 0 stays zero
    assert np.all(oracle.norm_rope(np.zeros((1, 1, 512)), eps=1e-6) == 0.0)


def test_norm_rope_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((5, 4, 512)) * rng.uniform(0.01, 100.0, (5, 4, 1))
    pos = rng.integers(0, 1 << 20, 5)
    y = oracle.norm_rope(x, eps=0.0, pos=pos, rope_base=10000.0)
    # the rotation keeps every pair's length, so the RMS stays 1
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-12)
    assert np.allclose(oracle.norm_rope(3.5 * x, eps=0.0, pos=pos, rope_base=10000.0), y, rtol=1e-12, atol=1e-12)
    # dims below 448 are untouched by the rotation
    y0 = oracle.norm_rope(x, eps=0.0)
    assert np.array_equal(y[..., :448], y0[..., :448])


def test_norm_rope_worked_angles():
    # position 1: pair 0 turns by exactly 1 rad, pair 16 by 10000^(-1/2) = 0.01 rad
    x = np.zeros((1, 1, 512))
    x[0, 0, 448] = 1.0          # (a, b) = (1, 0) for pair 0
    x[0, 0, 480 + 16] = 1.0     # (a, b) = (0, 1) for pair 16
    y = oracle.norm_rope(x, eps=0.0, pos=[1], rope_base=10000.0)[0, 0] / np.sqrt(256.0)
    assert abs(y[448] - 0.5403023058681398) < 1e-15 and abs(y[480] - 0.8414709848078965) < 1e-15
    # (0, 1) -> (-sin, cos) at 0.01 rad
    assert abs(y[448 + 16] + 0.009999833334166664) < 1e-15 and abs(y[480 + 16] - 0.9999500004166653) < 1e-15
    # position 0 rotates nothing
    y0 = oracle.norm_rope(x, eps=0.0, pos=[0], rope_base=10000.0)
    assert np.array_equal(y0, oracle.norm_rope(x, eps=0.0))


def test_norm_rope_relative_positions():
    # dot(rope(q, t), rope(k, s)) depends on t - s only, and equals the
    # unrotated dot product at t = s
    rng = np.random.default_rng(42)
    q = rng.standard_normal((1, 1, 512))
    k = rng.standard_normal((1, 1, 512))

    def dot(t, s):
        a = oracle.norm_rope(q, eps=0.0, pos=[t], rope_base=10000.0)[0, 0]
        b = oracle.norm_rope(k, eps=0.0, pos=[s], rope_base=10000.0)[0, 0]
        return float(a @ b)

    base = float(oracle.norm_rope(q, eps=0.0)[0, 0] @ oracle.norm_rope(k, eps=0.0)[0, 0])
    assert abs(dot(5000, 5000) - base) < 1e-9
    assert abs(dot(700, 200) - dot(10700, 10200)) < 1e-9
    assert abs(dot(700, 200) - base) > 1e-3


def test_norm_rope_inverts_the_output_rotation():
    # one key, rotated forward at position t, attended by a query at t: the
    # softmax weight is 1, so the output is the key, rotated back to where it was
    rng = np.random.default_rng(43)
    t = 777777
    k = rng.standard_normal((1, 1, 512))
    kn = oracle.norm_rope(k, eps=1e-6)
    kr = oracle.norm_rope(k, eps=1e-6, pos=[t], rope_base=10000.0)
    qb, _ = _q_and_keys(44, 1)
    o, _ = oracle.attention(qb, 1.0, kr.reshape(1, 512), rope_base=10000.0, t=t)
    assert np.allclose(o, np.broadcast_to(kn.reshape(1, 512), (64, 512)), rtol=0, atol=2e-6)
