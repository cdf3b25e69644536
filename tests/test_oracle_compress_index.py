"""Pins of the oracle's compressor and lightning-indexer score.

Anchors: closed forms (m = 1 identity, m = 2 sigmoid form, equal scores give
the mean), special inputs that isolate each term of the score (one head, one
dimension, ReLU cut, per-head weight, key scale) and invariances.
"""
import numpy as np
import torch

import oracle
from compressed_sparse_attention_layer_gb300 import synth


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- compressor
def test_compress_m1_is_identity():
    C = synth.normal_bf16(synth.stream_id(1, 1), 0, 64 * 512).reshape(64, 512)
    Z = synth.normal_bf16(synth.stream_id(1, 2), 0, 64 * 512).reshape(64, 512)
    b = synth.normal_f32(synth.stream_id(1, 3), 0, 512, sigma=0.1).reshape(1, 512)
    e = oracle.compress(C, Z, b, 1)
    assert np.array_equal(e, _f(C).astype(np.float32))


def test_compress_m2_closed_form():
    n = 256
    C = synth.normal_bf16(synth.stream_id(2, 1), 0, n * 512).reshape(n, 512)
    Z = synth.normal_bf16(synth.stream_id(2, 2), 0, n * 512).reshape(n, 512)
    b = synth.normal_f32(synth.stream_id(2, 3), 0, 1024, sigma=0.1).reshape(2, 512)
    e = oracle.compress(C, Z, b, 2)
    c = _f(C).reshape(n // 2, 2, 512)
    a = _f(Z).reshape(n // 2, 2, 512) + b.astype(np.float64)[None]
    w0 = 1.0 / (1.0 + np.exp(a[:, 1] - a[:, 0]))           # two-way softmax = logistic
    want = w0 * c[:, 0] + (1.0 - w0) * c[:, 1]
    assert np.allclose(e, want, rtol=1e-6, atol=1e-7)
    assert e.shape == (n // 2, 512)


def test_compress_equal_scores_give_mean_and_dominance():
    C = synth.normal_bf16(synth.stream_id(3, 1), 0, 8 * 512).reshape(8, 512)
    Z = np.zeros((8, 512), np.uint16)
    e = oracle.compress(C, Z, np.zeros((2, 512), np.float32), 2)
    c = _f(C).reshape(4, 2, 512)
    assert np.array_equal(e, ((c[:, 0] + c[:, 1]) / 2).astype(np.float32))
    Zd = np.zeros((8, 512), np.float32)
    Zd[0::2] = 60.0
    Zd[1::2] = -60.0
    e = oracle.compress(C, _bf16(Zd), np.zeros((2, 512), np.float32), 2)
    # a score gap of 120 leaves the other member a weight of e^-120: below fp32 resolution
    assert np.array_equal(e, c[:, 0].astype(np.float32))
    # the bias is indexed by offset in the group: a bias favouring offset 1 flips it
    bias = np.zeros((2, 512), np.float32)
    bias[1] = 200.0
    e = oracle.compress(C, _bf16(Zd), bias, 2)
    assert np.array_equal(e, c[:, 1].astype(np.float32))


def test_compress_tail_and_group_symmetry():
    C = synth.normal_bf16(synth.stream_id(4, 1), 0, 9 * 512).reshape(9, 512)
    Z = synth.normal_bf16(synth.stream_id(4, 2), 0, 9 * 512).reshape(9, 512)
    b = synth.normal_f32(synth.stream_id(4, 3), 0, 1024, sigma=0.1).reshape(2, 512)
    e = oracle.compress(C, Z, b, 2)
    assert e.shape == (4, 512)          # the ninth token waits for its partner
    # swapping the two members of each pair together with the bias rows changes nothing
    perm = np.arange(8).reshape(4, 2)[:, ::-1].reshape(-1)
    e2 = oracle.compress(C[:8][perm], Z[:8][perm], b[::-1].copy(), 2)
    assert np.allclose(e, e2, rtol=1e-7, atol=0)


# ---------------------------------------------------------------- indexer
def _keys(n, seed):
    x = synth.normal_f32(synth.stream_id(seed, 9), 0, n * 128).reshape(n, 128)
    return oracle.quant_fp8(x)


def test_index_score_isolates_one_term():
    codes, scales = _keys(64, 21)
    kval = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy() * scales[:, None]
    for h, d in [(0, 0), (5, 17), (31, 127)]:
        qi = np.zeros((32, 128), np.float32)
        qi[h, d] = 1.0
        w = np.zeros(32, np.float32)
        w[h] = 1.0
        s = oracle.index_scores(_bf16(qi), w, codes, scales)
        assert np.array_equal(s, np.maximum(kval[:, d], 0.0))           # ReLU(k_d)
        qi[h, d] = -1.0
        s = oracle.index_scores(_bf16(qi), w, codes, scales)
        assert np.array_equal(s, np.maximum(-kval[:, d], 0.0))          # sign follows q
        w[h] = 0.0
        assert not oracle.index_scores(_bf16(qi), w, codes, scales).any()


def test_index_score_weights_heads_and_scale():
    codes, scales = _keys(128, 22)
    qi = synth.normal_bf16(synth.stream_id(22, 1), 0, 4096).reshape(32, 128)
    w = synth.uniform_f32(synth.stream_id(22, 2), 0, 32)
    s = oracle.index_scores(qi, w, codes, scales)
    # per-head weights enter linearly
    assert np.array_equal(oracle.index_scores(qi, w * np.float32(4.0), codes, scales), 4.0 * s)
    # the sum over heads: two disjoint halves of the weights add up
    wa, wb = w.copy(), w.copy()
    wa[16:] = 0
    wb[:16] = 0
    sa = oracle.index_scores(qi, wa, codes, scales)
    sb = oracle.index_scores(qi, wb, codes, scales)
    assert np.allclose(sa + sb, s, rtol=1e-13, atol=0)
    # permuting heads of q and w together changes nothing
    p = np.random.default_rng(0).permutation(32)
    assert np.allclose(oracle.index_scores(qi[p], w[p], codes, scales), s, rtol=1e-13, atol=0)
    # the key's fp32 scale multiplies the score
    assert np.array_equal(oracle.index_scores(qi, w, codes, scales * np.float32(2.0)), 2.0 * s)
    # all heads see the ReLU: negating q keeps only the other half-space
    sn = oracle.index_scores((qi ^ np.uint16(0x8000)), w, codes, scales)
    assert (s >= 0).all() and (sn >= 0).all()
    assert ((s > 0) | (sn > 0)).all()


def test_index_scores_positions_gather():
    codes, scales = _keys(100, 23)
    qi = synth.normal_bf16(synth.stream_id(23, 1), 0, 4096).reshape(32, 128)
    w = synth.uniform_f32(synth.stream_id(23, 2), 0, 32)
    s = oracle.index_scores(qi, w, codes, scales)
    pos = np.array([99, 0, 50, 50, 7], np.int32)
    assert np.array_equal(oracle.index_scores(qi, w, codes, scales, positions=pos), s[pos])
