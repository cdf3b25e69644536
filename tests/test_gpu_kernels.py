"""Parity of each CUDA entry point against the CPU oracle (needs a GPU).

Bit-exact: quantisers, Top-K given identical scores, pool construction.
Tolerances (floating point): compressor rounds once from double precision on
both sides; indexer scores rel 1e-5 -- the scan splits each head of the bf16
query into two e4m3 parts, hi = e4m3(q 2^-e) and lo = e4m3(q 2^-e - hi) with
max|q 2^-e| in [128, 256): an element within about 2^-10 of its head's
largest keeps its bf16 value exactly, a smaller one is carried to an absolute
error of at most 2^-17 of that largest element (lo's subnormal step); the
products of the key codes with hi and lo accumulate in fp32 on the tensor
cores, against the oracle's double precision; attention max-abs 2e-3 and
rel-L2 1e-3 given identical indices.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_layer_gb300 import csa2, synth
from compressed_sparse_attention_layer_gb300.device import DeviceWorkload
from compressed_sparse_attention_layer_gb300 import workloads as W
from tests.reference import SeqOracle, attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from compressed_sparse_attention_layer_gb300 import build
    build.build()
    csa2.load()


def _special_rows(n_rows, dim, seed):
    """Random rows plus rows built to hit ties, signed zeros, subnormals and saturation."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n_rows, dim)) * np.exp(rng.uniform(-6, 6, (n_rows, 1)))).astype(np.float32)
    # MXFP4 ties: blocks whose amax is 6 contain every grid midpoint
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.9, 0.5, 3.0, 0.1], np.float32)
    x[0, :mids.size] = mids
    x[0, 16:16 + mids.size] = -mids
    x[1] = 0.0
    x[1, 3] = -0.0
    x[2, :] = np.float32(1e-41)              # subnormal block maxima
    x[2, 5] = np.float32(-3e-42)
    x[3, :] = np.float32(3e38)               # huge values
    x[3, 7] = np.float32(-1.7e38)
    x[4, :] = -0.0
    x[5, ::2] = np.float32(2.0 ** -130)
    return x


def test_quant_mxfp4_bit_exact():
    x = _special_rows(300, 512, 1)
    codes, scales = oracle.quant_mxfp4(x)
    xd = torch.from_numpy(x).cuda()
    gc = torch.zeros((320, 256), dtype=torch.uint8, device="cuda")
    gs = torch.zeros((320, 16), dtype=torch.uint8, device="cuda")
    csa2.csa2_quant_mxfp4(xd, gc, gs)
    torch.cuda.synchronize()
    assert np.array_equal(gc[:300].cpu().numpy(), codes)
    assert np.array_equal(gs[:300].cpu().numpy(), scales)
    # slot mapping: scattered destinations, negative slots skipped
    perm = np.random.default_rng(2).permutation(320)[:300].astype(np.int64)
    perm[7] = -1
    gc.zero_()
    gs.zero_()
    csa2.csa2_quant_mxfp4(xd, gc, gs, slots=torch.from_numpy(perm).cuda())
    torch.cuda.synchronize()
    got_c, got_s = gc.cpu().numpy(), gs.cpu().numpy()
    keep = perm >= 0
    assert np.array_equal(got_c[perm[keep]], codes[keep]) and np.array_equal(got_s[perm[keep]], scales[keep])


def test_quant_fp4_e4m3_bit_exact():
    """FP4 with one E4M3 scale per 16 elements: bit-exact against the oracle,
    including huge values (scale saturating at 448), signed zeros, subnormal
    inputs (scale rounding to zero) and scattered destination slots."""
    x = _special_rows(300, 512, 3)
    x[6, :16] = 1.0
    x[6, 16:32] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -6.0, 0.0, -0.0, 3.0, 4.0, 1.5, 0.5, 2.0]
    codes, scales = oracle.quant_fp4_e4m3(x)
    xd = torch.from_numpy(x).cuda()
    gc = torch.zeros((320, 256), dtype=torch.uint8, device="cuda")
    gs = torch.zeros((320, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_quant_fp4_e4m3(xd, gc, gs)
    torch.cuda.synchronize()
    assert np.array_equal(gc[:300].cpu().numpy(), codes)
    assert np.array_equal(gs[:300].cpu().numpy(), scales)
    perm = np.random.default_rng(4).permutation(320)[:300].astype(np.int64)
    perm[9] = -1
    gc.zero_()
    gs.zero_()
    csa2.csa2_quant_fp4_e4m3(xd, gc, gs, slots=torch.from_numpy(perm).cuda())
    torch.cuda.synchronize()
    got_c, got_s = gc.cpu().numpy(), gs.cpu().numpy()
    keep = perm >= 0
    assert np.array_equal(got_c[perm[keep]], codes[keep]) and np.array_equal(got_s[perm[keep]], scales[keep])


@pytest.mark.parametrize("dim", [128, 512])
def test_quant_fp8_bit_exact(dim):
    x = _special_rows(257, dim, 3 + dim)
    x[6, :] = 0.0
    x[7, :] = np.float32(448.0)
    x[8, :] = np.linspace(-1, 1, dim, dtype=np.float32)
    codes, scales = oracle.quant_fp8(x)
    gc = torch.zeros((257, dim), dtype=torch.uint8, device="cuda")
    gs = torch.zeros((257,), dtype=torch.float32, device="cuda")
    csa2.csa2_quant_fp8(torch.from_numpy(x).cuda(), gc, gs)
    torch.cuda.synchronize()
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    got = gc.cpu().numpy()
    bad = np.argwhere(got != codes)
    assert bad.size == 0, (bad[:5], x[tuple(bad[0])], got[tuple(bad[0])], codes[tuple(bad[0])])


@pytest.mark.parametrize("m", [1, 2, 4])
def test_compress_matches_oracle(m):
    n_tok = 1000 * m + (m - 1)
    C = synth.normal_bf16(synth.stream_id(50, 1), 0, n_tok * 512).reshape(n_tok, 512)
    Z = synth.normal_bf16(synth.stream_id(50, 2), 0, n_tok * 512).reshape(n_tok, 512)
    bias = synth.normal_f32(synth.stream_id(50, 3), 0, m * 512, sigma=0.1).reshape(m, 512)
    want = oracle.compress(C, Z, bias, m)
    out = torch.empty((n_tok // m, 512), dtype=torch.float32, device="cuda")
    t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    csa2.csa2_compress(t(C), t(Z), torch.from_numpy(bias).cuda(), m, out)
    got = out.cpu().numpy()
    # both sides round once from double precision: differences need a last-bit exp tie
    diff = got.view(np.uint32) != want.view(np.uint32)
    assert diff.mean() <= 1e-5, diff.sum()
    assert np.allclose(got, want, rtol=2e-7, atol=0)


@pytest.mark.parametrize("kv_format,m", [(0, 1), (0, 4), (1, 2)])
def test_append_entries_matches_the_separate_calls(kv_format, m):
    """csa2_append_entries: the compressor, the main-KV quantiser of the cache's
    format and the indexer key's FP8 quantiser in one launch, bit for bit the
    results of csa2_compress + csa2_quant_mxfp4 / _fp4_e4m3 + csa2_quant_fp8 at
    scattered slots (one skipped, one past the cache and flagged), and the
    quantised codes equal to the oracle's of the entries it returns."""
    n_ent = 300
    n_tok = n_ent * m + (m - 1)                    # a trailing partial group is not compressed
    C = synth.normal_bf16(synth.stream_id(51, 1, m), 0, n_tok * 512).reshape(n_tok, 512)
    Z = synth.normal_bf16(synth.stream_id(51, 2, m), 0, n_tok * 512).reshape(n_tok, 512)
    bias = synth.normal_f32(synth.stream_id(51, 3, m), 0, m * 512, sigma=0.1).reshape(m, 512)
    ik = _special_rows(n_ent, 128, 9 + m)
    bt = torch.zeros((1, 8), dtype=torch.int32)
    caches = [csa2.PagedCache(8, bt, "cuda", kv_format=kv_format) for _ in range(2)]
    S = caches[0].num_slots
    slots = np.random.default_rng(12 + m).permutation(S)[:n_ent].astype(np.int64)
    slots[5] = -1
    slots[6] = S + 3
    t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    Cd, Zd, bd, ikd = t(C), t(Z), torch.from_numpy(bias).cuda(), torch.from_numpy(ik).cuda()
    sd = torch.from_numpy(slots).cuda()
    entries = torch.full((n_ent, 512), float("nan"), dtype=torch.float32, device="cuda")
    csa2.csa2_append_entries(caches[0].struct(), Cd, Zd, bd, m, ikd, slots=sd, entries=entries)
    ref = caches[1]
    e = torch.empty((n_ent, 512), dtype=torch.float32, device="cuda")
    csa2.csa2_compress(Cd, Zd, bd, m, e)
    quant = csa2.csa2_quant_fp4_e4m3 if kv_format == csa2.KV_FP4_E4M3 else csa2.csa2_quant_mxfp4
    quant(e, ref.kv_codes, ref.kv_scales, slots=sd, status=ref.status)
    csa2.csa2_quant_fp8(ikd, ref.ik_codes, ref.ik_scales, slots=sd, status=ref.status)
    torch.cuda.synchronize()
    got, want = caches[0], ref
    assert np.array_equal(entries.cpu().numpy().view(np.uint32), e.cpu().numpy().view(np.uint32))
    for name in ("kv_codes", "kv_scales", "ik_codes"):
        assert torch.equal(getattr(got, name), getattr(want, name)), name
    assert torch.equal(got.ik_scales.view(torch.int32), want.ik_scales.view(torch.int32))
    assert int(got.status[0]) == csa2.DEV_BAD_SLOT == int(want.status[0])
    # against the oracle: the codes at the written slots
    keep = (slots >= 0) & (slots < S)
    oq = oracle.quant_fp4_e4m3 if kv_format == csa2.KV_FP4_E4M3 else oracle.quant_mxfp4
    codes, scales = oq(entries.cpu().numpy())
    assert np.array_equal(got.kv_codes.cpu().numpy()[slots[keep]], codes[keep])
    assert np.array_equal(got.kv_scales.cpu().numpy()[slots[keep]], scales[keep])
    icodes, iscales = oracle.quant_fp8(ik)
    assert np.array_equal(got.ik_codes.cpu().numpy()[slots[keep]], icodes[keep])
    assert np.array_equal(got.ik_scales.cpu().numpy()[slots[keep]].view(np.uint32), iscales[keep].view(np.uint32))
    # untouched slots keep their contents
    untouched = np.setdiff1d(np.arange(S), slots[keep])
    assert not got.kv_codes.cpu().numpy()[untouched].any()


def _dw(wl, **kw):
    return DeviceWorkload(wl, **kw)


def test_index_scores_decode_small():
    wl = W.decode_small()
    dw = _dw(wl)
    so = SeqOracle(wl, 0)
    ld = (wl.max_entries + 7) // 8 * 8
    scores = torch.full((1, ld), np.nan, dtype=torch.float32, device="cuda")
    bmax = torch.full((1, ld // 8), np.nan, dtype=torch.float32, device="cuda")
    nvis = torch.zeros((1,), dtype=torch.int32, device="cuda")
    csa2.csa2_index_scores(dw.cstruct, dw.batch, dw.qi[0], dw.w[0], scores, bmax, nvis, ld)
    torch.cuda.synchronize()
    want = so.scores(0, 0, np.arange(wl.entries(0)))
    got = scores[0].cpu().numpy().astype(np.float64)
    assert int(nvis[0]) == wl.entries(0)
    assert np.allclose(got, want, rtol=1e-5, atol=1e-5 * np.abs(want).max())
    assert np.array_equal(bmax[0].cpu().numpy(), scores[0].cpu().numpy().reshape(-1, 8).max(axis=1))
    assert int(dw.cache.status[0]) == 0


def test_topk_bit_exact_given_scores():
    rng = np.random.default_rng(9)
    rows, ld = 6, 50000
    s = rng.integers(0, 300, (rows, ld)).astype(np.float32) * np.float32(0.5)     # heavy ties
    s[1] = -s[1]
    s[2, :100] = -0.0
    s[2, 100:] = -1.0
    lens = np.array([50000, 49999, 40000, 600, 512, 3], np.int32)
    cand = np.sort(rng.choice(10 ** 6, (rows, ld)), axis=1).astype(np.int32)
    for use_cand in (False, True):
        out = torch.empty((rows, 512), dtype=torch.int32, device="cuda")
        csa2.csa2_topk(torch.from_numpy(s).cuda(), torch.from_numpy(lens).cuda(), 512, out,
                       cand=torch.from_numpy(cand).cuda() if use_cand else None)
        got = out.cpu().numpy()
        for r in range(rows):
            n = lens[r]
            want = oracle.topk(s[r, :n].astype(np.float64), cand[r, :n] if use_cand else None)
            assert np.array_equal(got[r], want), (r, use_cand)


def test_topk_rows_of_at_most_16384_bit_exact():
    """Rows that fit one CTA (the pool Top-512 path): heavy ties, -0.0 / +0.0,
    -inf, fewer valid slots than k, exactly k, one, none; with and without cand."""
    rng = np.random.default_rng(19)
    rows, ld = 9, 16384
    s = rng.integers(0, 200, (rows, ld)).astype(np.float32) * np.float32(0.25)
    s[1] = -s[1]
    s[2, ::2] = -0.0
    s[2, 1::2] = 0.0
    s[3, :] = 7.0                                              # all equal: lowest slots win
    s[4, 5000:] = -np.inf
    s[5] = rng.standard_normal(ld).astype(np.float32)          # distinct values
    lens = np.array([16384, 16383, 16384, 16384, 9000, 513, 512, 1, 0], np.int32)
    cand = np.sort(rng.choice(10 ** 6, (rows, ld)), axis=1).astype(np.int32)
    for use_cand in (False, True):
        out = torch.full((rows, 512), -7, dtype=torch.int32, device="cuda")
        csa2.csa2_topk(torch.from_numpy(s).cuda(), torch.from_numpy(lens).cuda(), 512, out,
                       cand=torch.from_numpy(cand).cuda() if use_cand else None)
        got = out.cpu().numpy()
        for r in range(rows):
            n = lens[r]
            want = oracle.topk(s[r, :n].astype(np.float64), cand[r, :n] if use_cand else None)
            assert np.array_equal(got[r], want), (r, use_cand)


def test_topk_rows_threshold_cases_bit_exact():
    """The one-CTA select's bound-and-radix path: distinct values (the k-th
    largest in a small bin, ranked directly), ties exactly at the k-th value,
    scores concentrated like the indexer's (positive, a narrow range), a row
    whose group maxima exclude almost everything, a negative row, and k larger
    than the 512 groups of the bound."""
    rng = np.random.default_rng(23)
    rows, ld = 6, 16384
    s = rng.standard_normal((rows, ld)).astype(np.float32)
    v = np.sort(s[1])[::-1][511]
    s[1, rng.choice(np.flatnonzero(s[1] < v), 5, replace=False)] = v       # ties at the threshold
    s[2] = (rng.gamma(2.0, 0.3, ld) * rng.uniform(0.9, 1.1, ld)).astype(np.float32) + np.float32(3.0)
    s[3] = np.float32(1.0)
    s[3, rng.choice(ld, 600, replace=False)] = rng.uniform(2.0, 3.0, 600).astype(np.float32)
    s[4] = -np.abs(s[4]) - np.float32(1.0)
    lens = np.array([16384, 16384, 16384, 16384, 16000, 16384], np.int32)
    for k in (512, 1500):
        out = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
        csa2.csa2_topk(torch.from_numpy(s).cuda(), torch.from_numpy(lens).cuda(), k, out)
        got = out.cpu().numpy()
        for r in range(rows):
            n = lens[r]
            want = oracle.topk(s[r, :n].astype(np.float64), None, k=k)
            assert np.array_equal(got[r], want), (r, k)


def test_topk_blocks_bit_exact():
    rng = np.random.default_rng(10)
    rows = 4
    nvis = np.array([1 << 20, 1000003, 16384 * 8 + 5, 9], np.int32)
    ld_b = (int(nvis.max()) + 7) // 8
    bm = rng.integers(0, 5000, (rows, ld_b)).astype(np.float32)
    pool = torch.full((rows, 16384), -7, dtype=torch.int32, device="cuda")
    plen = torch.zeros((rows,), dtype=torch.int32, device="cuda")
    csa2.csa2_topk_blocks(torch.from_numpy(bm).cuda(), torch.from_numpy(nvis).cuda(), 2048, pool, plen)
    got, gl = pool.cpu().numpy(), plen.cpu().numpy()
    for r in range(rows):
        n = int(nvis[r])
        scores = np.repeat(bm[r, :(n + 7) // 8].astype(np.float64), 8)[:n]   # block max = that value
        want = oracle.block_pool(scores, n)
        assert gl[r] == want.size and np.array_equal(got[r, :gl[r]], want), r


def test_topk_blocks_single_stage_bit_exact():
    """Rows of at most 16,384 blocks (one select per row): ties, fewer blocks
    than the pool holds, a partial last block."""
    rng = np.random.default_rng(11)
    nvis = np.array([131072, 131067, 70000, 16384, 100, 0], np.int32)
    rows = nvis.size
    ld_b = 16384
    bm = rng.integers(0, 300, (rows, ld_b)).astype(np.float32)
    pool = torch.full((rows, 16384), -7, dtype=torch.int32, device="cuda")
    plen = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    csa2.csa2_topk_blocks(torch.from_numpy(bm).cuda(), torch.from_numpy(nvis).cuda(), 2048, pool, plen)
    got, gl = pool.cpu().numpy(), plen.cpu().numpy()
    for r in range(rows):
        n = int(nvis[r])
        scores = np.repeat(bm[r, :(n + 7) // 8].astype(np.float64), 8)[:n]
        want = oracle.block_pool(scores, n)
        assert gl[r] == want.size and np.array_equal(got[r, :gl[r]], want), r


@pytest.mark.parametrize("schedule", [csa2.ATTN_SCHEDULE_CHUNKS, csa2.ATTN_SCHEDULE_ROWS])
def test_sparse_attn_given_oracle_indices(schedule):
    """Both attention schedules (one cluster per key chunk and a merge; one
    persistent cluster per row with an online softmax) on the oracle's
    selection, a padded one, the window alone, and selections of k = 200 and
    k = 1 (a partial chunk, one chunk plus the window)."""
    wl = W.decode_small()
    dw = _dw(wl)
    dw.attn_options = dict(flags=schedule)
    so = SeqOracle(wl, 0)
    idx, pool, _ = so.full(0, 0)
    o_ref, lse_ref = so.attention(0, 0, idx)
    o = torch.empty((1, 64, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, 64), dtype=torch.float32, device="cuda")
    ws_n = csa2.csa2_sparse_attn_workspace_size(1, 1)
    ws = torch.empty((max(ws_n, 256),), dtype=torch.uint8, device="cuda")
    csa2.csa2_sparse_attn(dw.cstruct, dw.batch, dw.q[0], 1.0, torch.from_numpy(idx[None]).cuda(), dw.swa(0),
                          o, lse, workspace=ws)
    ok, info = attn_close(o[0].cpu().numpy(), lse[0].cpu().numpy(), o_ref, lse_ref)
    assert ok, info
    for kk in (200, 1):
        sub = np.ascontiguousarray(idx[:kk])
        o_ref_k, lse_ref_k = so.attention(0, 0, sub)
        csa2.csa2_sparse_attn(dw.cstruct, dw.batch, dw.q[0], 1.0, torch.from_numpy(sub[None]).cuda(), dw.swa(0),
                              o, lse, workspace=ws)
        ok, info = attn_close(o[0].cpu().numpy(), lse[0].cpu().numpy(), o_ref_k, lse_ref_k)
        assert ok, (kk, info)
    assert int(dw.cache.status[0]) == 0
    # a shorter, padded selection (-1 slots) and the window alone
    idx2 = idx.copy()
    idx2[100:] = -1
    o_ref2, lse_ref2 = so.attention(0, 0, idx2)
    csa2.csa2_sparse_attn(dw.cstruct, dw.batch, dw.q[0], 1.0, torch.from_numpy(idx2[None]).cuda(), dw.swa(0),
                          o, lse, workspace=ws)
    ok, info = attn_close(o[0].cpu().numpy(), lse[0].cpu().numpy(), o_ref2, lse_ref2)
    assert ok, info
    idx3 = np.full_like(idx, -1)
    o_ref3, lse_ref3 = so.attention(0, 0, idx3)
    csa2.csa2_sparse_attn(dw.cstruct, dw.batch, dw.q[0], 1.0, torch.from_numpy(idx3[None]).cuda(), dw.swa(0),
                          o, lse, workspace=ws)
    ok, info = attn_close(o[0].cpu().numpy(), lse[0].cpu().numpy(), o_ref3, lse_ref3)
    assert ok, info


def test_device_generator_matches_host():
    s = synth.stream_id(3, 4, 5)
    for start, count in [(0, 100000), ((1 << 32) - 500, 1000)]:
        a = synth.normal_bf16(s, start, count)
        b = synth.normal_bf16_torch(s, start, count, "cuda").view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(a, b)
        assert np.array_equal(synth.uniform_f32(s, start, count),
                              synth.uniform_f32_torch(s, start, count, "cuda").cpu().numpy())


def test_bad_page_ids_are_flagged_not_read():
    wl = W.decode_small()
    dw = _dw(wl)
    dw.cache.block_table[0, 3] = 10 ** 6          # outside the cache
    dw.cache.block_table[0, 5] = -4
    dw.cstruct = dw.cache.struct()
    dw.run_layer(0)
    torch.cuda.synchronize()
    assert int(dw.cache.status[0]) & csa2.DEV_BAD_PAGE
    assert torch.isfinite(dw.o[0]).all()


def _index_rows(dw, ld):
    rows = dw.rows
    scores = torch.full((rows, ld), np.nan, dtype=torch.float32, device="cuda")
    bmax = torch.full((rows, ld // 8), np.nan, dtype=torch.float32, device="cuda")
    nvis = torch.zeros((rows,), dtype=torch.int32, device="cuda")
    l = dw.wl.layers.index("full")
    csa2.csa2_index_scores(dw.cstruct, dw.batch, dw.qi[l], dw.w[l], scores, bmax, nvis, ld)
    torch.cuda.synchronize()
    return scores.cpu().numpy(), bmax.cpu().numpy(), nvis.cpu().numpy()


def test_index_scores_ragged_and_extreme_heads():
    """Ragged rows (persistent work list) and indexer-query heads spanning
    2^-60 .. 2^60 in magnitude (the per-head power-of-two scaling)."""
    wl = W.Workload("ragged_ix", 61, 4, [1000, 70001, 130, 9], 1, ["full"])
    dw = _dw(wl)
    mult = np.exp2(np.linspace(-60, 60, 32)).astype(np.float32)
    for b in range(wl.batch):
        qi = synth.bf16_bits_to_f32(wl.qi_bits(0, b)[0]) * mult[:, None]
        bits = torch.from_numpy(qi).to(torch.bfloat16)
        dw.qi[0][b].copy_(bits.cuda())
    ld = (wl.max_entries + 7) // 8 * 8
    s, bm, nv = _index_rows(dw, ld)
    for b in range(wl.batch):
        so = SeqOracle(wl, b)
        E = wl.entries(b)
        assert nv[b] == E
        qib = dw.qi[0][b].cpu().view(torch.int16).numpy().view(np.uint16)
        codes, scales = so.ik()
        want = oracle.index_scores(qib, wl.w(0, b)[0], codes, scales)
        got = s[b, :E].astype(np.float64)
        assert np.allclose(got, want, rtol=1e-5, atol=1e-6 * np.abs(want).max()), b
        nb = (E + 7) // 8
        pad = np.full(nb * 8, -np.inf, np.float32)
        pad[:E] = s[b, :E]
        assert np.array_equal(bm[b, :nb], pad.reshape(nb, 8).max(axis=1)), b


def test_index_scores_many_query_rows_causal():
    """More than 256 query rows (one grid row per query) with causal visibility."""
    wl = W.Workload("causal_ix", 62, 1, [6000], 1, ["full"], nq=300, prefill_new=300, swa_rows=300 + 128)
    dw = _dw(wl)
    ld = (wl.max_entries + 7) // 8 * 8
    s, bm, nv = _index_rows(dw, ld)
    so = SeqOracle(wl, 0)
    for i in (0, 1, 137, 299):
        t, nvis = so.visible(i)
        assert nv[i] == nvis == t + 1
        want = so.scores(0, i, np.arange(nvis))
        assert np.allclose(s[i, :nvis], want, rtol=1e-5, atol=1e-6 * np.abs(want).max()), i


def test_index_scores_pool_gathered():
    """Reindex rescoring of a scattered candidate pool (incl. a ragged tail and an
    out-of-range position, which is flagged and scored -inf)."""
    wl = W.Workload("pool_ix", 63, 3, [50000, 9000, 70000], 1, ["full"])
    dw = _dw(wl)
    rng = np.random.default_rng(63)
    ld = 16384
    pool = np.full((3, ld), -1, np.int32)
    lens = np.array([16384, 1000, 7], np.int32)
    for b in range(3):
        blocks = np.sort(rng.choice(wl.entries(b) // 8, lens[b] // 8 + 1, replace=False))
        pos = (blocks[:, None] * 8 + np.arange(8)).reshape(-1)[:lens[b]]
        pool[b, :lens[b]] = pos
    pool[2, 3] = wl.entries(2) + 5            # beyond the context
    scores = torch.full((3, ld), np.nan, dtype=torch.float32, device="cuda")
    csa2.csa2_index_scores_pool(dw.cstruct, dw.batch, dw.qi[0], dw.w[0], torch.from_numpy(pool).cuda(),
                                torch.from_numpy(lens).cuda(), scores)
    torch.cuda.synchronize()
    got = scores.cpu().numpy()
    for b in range(3):
        so = SeqOracle(wl, b)
        ok = (pool[b, :lens[b]] >= 0) & (pool[b, :lens[b]] < wl.entries(b))
        want = so.scores(0, 0, pool[b, :lens[b]][ok])
        assert np.allclose(got[b, :lens[b]][ok], want, rtol=1e-5, atol=1e-6 * np.abs(want).max()), b
        assert np.all(np.isneginf(got[b, :lens[b]][~ok]))
        assert np.all(np.isnan(got[b, lens[b]:]))
    assert int(dw.cache.status[0]) & csa2.DEV_BAD_INDEX


def _norm_rope_tol(ref):
    """Per-element bound for the fp32 kernel against the fp64 oracle: the
    fp32 mean square (16 products per lane, a 5-level shuffle tree) and the
    scale carry <= ~1e-6 relative; the rotation adds the fp32 angle and
    sin / cos errors (<= 3e-7 absolute) times the pair's size.  So 4e-6 times
    |y_d| outside the RoPE dims and times |y_448+i| + |y_480+i| inside them."""
    mag = np.abs(ref).copy()
    pair = np.abs(ref[..., 448:480]) + np.abs(ref[..., 480:512])
    mag[..., 448:480] = pair
    mag[..., 480:512] = pair
    return 4e-6 * mag


@pytest.mark.parametrize("rows,vecs,rope_base,use_gamma", [(37, 64, 10000.0, True), (1000, 1, 10000.0, False),
                                                            (5, 3, 0.0, True), (1, 64, 1e6, False)])
def test_norm_rope_matches_oracle(rows, vecs, rope_base, use_gamma):
    rng = np.random.default_rng(rows * 100 + vecs)
    x = (rng.standard_normal((rows, vecs, 512)) * np.exp(rng.uniform(-6, 6, (rows, vecs, 1)))).astype(np.float32)
    x[0, 0] = 0.0                                           # zero vector: stays zero (eps > 0)
    pos = rng.integers(0, 1 << 20, rows).astype(np.int64)
    pos[0] = 0
    pos[-1] = (1 << 20) - 1
    gamma = rng.uniform(0.5, 1.5, 512).astype(np.float32) if use_gamma else None
    eps = 1e-6
    ref = oracle.norm_rope(x, gamma, eps, pos, rope_base)
    tol = _norm_rope_tol(ref)
    xd = torch.from_numpy(x).cuda()
    gd = None if gamma is None else torch.from_numpy(gamma).cuda()
    pd = torch.from_numpy(pos).cuda()
    out = torch.empty_like(xd)
    csa2.csa2_norm_rope(xd, out, gd, eps, pd, rope_base)
    ob = torch.empty(xd.shape, dtype=torch.bfloat16, device="cuda")
    csa2.csa2_norm_rope(xd, ob, gd, eps, pd, rope_base)
    torch.cuda.synchronize()
    y = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y - ref) <= tol), float(np.max(np.abs(y - ref) - tol))
    assert np.all(y[0, 0] == 0.0)
    # bf16 output: the same values rounded once more (half an ulp of bf16 = 2^-8 relative)
    yb = ob.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yb - ref) <= 2.0 ** -8 * np.abs(ref) + tol)
    # in place (out = x) gives the same bits as out of place
    csa2.csa2_norm_rope(xd, xd, gd, eps, pd, rope_base)
    torch.cuda.synchronize()
    assert torch.equal(xd, out)


def test_norm_rope_empty_and_bad_arguments():
    x = torch.zeros((0, 64, 512), device="cuda")
    csa2.csa2_norm_rope(x, torch.empty_like(x), None, 1e-6, None, 10000.0)     # rows = 0: nothing to do
    x = torch.ones((2, 1, 512), device="cuda")
    with pytest.raises(csa2.Csa2Error):
        csa2.csa2_norm_rope(x, torch.empty_like(x), None, 1e-6, None, 10000.0)  # rope without positions
    with pytest.raises(csa2.Csa2Error):
        csa2.csa2_norm_rope(x, torch.empty_like(x), None, -1.0, None, 0.0)      # negative eps


def _prologue_gamma():
    """The RMSNorm weight of the benchmark's prologue workload (host generator)."""
    return (1.0 + 0.1 * synth.normal_f32(7101, 0, 512)).astype(np.float32)


def _norm_rope_full_size_check(out_rows, picks, H):
    """The oracle on the sampled vectors of the full-size prologue (inputs from
    the host generator) against the kernel's bf16 rows out_rows
    [len(picks)][512]: bf16 rounding plus the fp32 bound of _norm_rope_tol."""
    x = np.stack([synth.normal_f32(7100, int(v) * 512, 512) for v in picks]).reshape(len(picks), 1, 512)
    pos = (65536 + np.asarray(picks) // H).astype(np.int64)
    ref = oracle.norm_rope(x, _prologue_gamma(), 1e-6, pos, 10000.0)[:, 0]
    return np.abs(out_rows - ref) <= 2.0 ** -8 * np.abs(ref) + _norm_rope_tol(ref)


def test_norm_rope_full_size_sampled():
    """The prologue in the launch the benchmark times (8,192 query tokens x 64
    heads of 512 fp32 dims, bf16 out, positions from 65,536, rope_base
    10,000): 512 sampled vectors, the first and last among them, against the
    oracle."""
    T, H = 8192, 64
    dev = torch.device("cuda")
    x = synth.normal_f32_torch(7100, 0, T * H * 512, dev).view(T, H, 512)
    rng = np.random.default_rng(8192)
    picks = rng.choice(T * H, 512, replace=False)
    picks[:2] = [0, T * H - 1]
    pos = torch.arange(65536, 65536 + T, dtype=torch.int64, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    csa2.csa2_norm_rope(x, out, torch.from_numpy(_prologue_gamma()).to(dev), 1e-6, pos, 10000.0)
    torch.cuda.synchronize()
    got = out.view(T * H, 512)[torch.from_numpy(picks).to(dev)].float().cpu().numpy().astype(np.float64)
    ok = _norm_rope_full_size_check(got, picks, H)
    assert ok.all(), int((~ok).sum())
