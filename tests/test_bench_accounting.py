"""The benchmark's algorithmic-work accounting (host only): the bytes a layer
mode must move per query token at the headline workload, the scan's bytes
per launch, and the prefill scan's FLOPs -- the units the roofline fractions
and the per-layer-mode figures are computed from."""
import bench
from compressed_sparse_attention_layer_gb300 import csa2
from compressed_sparse_attention_layer_gb300 import workloads as W


def test_constants_match_the_library_binding():
    assert bench.KV_SCALE_BYTES == {csa2.KV_MXFP4: 16, csa2.KV_FP4_E4M3: 32} == csa2.KV_SCALE_BYTES
    assert bench.POOL_MAX == csa2.POOL_MAX == 2048 * 8


def test_decode_1m_bytes_per_query_token():
    wl = W.decode_1m()
    E = 1 << 20
    per_token = {m: v / 8 for m, v in bench.layer_bytes(wl).items()}
    attn = 512 * 272 + 128 * 516 + 65536 + 131072 + 256          # gathered KV, window, q, o, lse
    assert attn == 402176
    # Full: every indexer key (132 B) once, the block maxima, qi and w, the attention
    assert per_token["full"] == E * 132 + (E // 8) * 4 + 8192 + 128 + attn == 139346816
    # Reindex: the pool's keys and scores, qi and w, the attention (~2.64 MB)
    assert per_token["reindex"] == 16384 * 136 + 8192 + 128 + attn == 2638720
    # Reuse: the indices and the attention (~0.40 MB)
    assert per_token["reuse"] == 2048 + attn == 404224
    stack = sum(bench.layer_bytes(wl)[m] for m in wl.layers) / 8
    assert abs(stack / 1e6 - 155.97) < 0.01                    # 1 Full + 4 Reindex + 15 Reuse


def test_scan_work_units():
    bound, work = bench.scan_work(W.decode_1m())
    assert bound == "hbm" and work == 8 * ((1 << 20) * 132 + (1 << 17) * 4 + 8320)
    # four query tokens per sequence: the keys are read once for all four
    bound, work4 = bench.scan_work(W.decode_multi(q=4))
    vis = bench.rows_visible(W.decode_multi(q=4))
    assert vis[:4] == [(1 << 20) - 3, (1 << 20) - 2, (1 << 20) - 1, 1 << 20]
    assert work4 == 8 * (1 << 20) * 132 + sum((v // 8) * 4 + 8320 for v in vis)
    # the prefill chunk is counted in e4m3 products: query row i (token 65,536 + i,
    # m = 2) sees (65,537 + i) // 2 entries
    bound, flops = bench.scan_work(W.prefill())
    assert bound == "tensor"
    assert flops == sum((65537 + i) // 2 for i in range(8192)) * 32 * 128 * 2


def test_e2e_copy_groups():
    """Every layer's inputs are copied in exactly once, the first IN_EARLY
    layers' before the step's kernels; every layer's outputs go out exactly
    once, in order, in pairs with the last layer alone."""
    for n in (1, 2, 3, 4, 5, 6, 8, 20):
        early, late, out = bench.e2e_groups(n)
        assert early + late == list(range(n))
        assert early == list(range(min(bench.IN_EARLY, n)))
        assert sum(out, []) == list(range(n))
        assert all(1 <= len(g) <= bench.OUT_GROUP for g in out)
        assert len(out[-1]) == 1
    early, late, out = bench.e2e_groups(20)
    assert early == [0, 1, 2, 3, 4] and len(out) == 11 and out[-2:] == [[18], [19]]
