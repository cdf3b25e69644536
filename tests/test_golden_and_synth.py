"""Constants and footprint arithmetic the pages fix, the layer grouping, and the
shared seeded input generator (host numpy vs torch twin)."""
import json
import os

import numpy as np
import torch

import oracle
from compressed_sparse_attention_layer_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _json(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_config_table_arithmetic():
    c = _json("config_table.json")
    assert c["pool_max_blocks"] * c["pool_block_positions"] == c["pool_max_candidates"] == 16384
    assert c["topk"] == oracle.TOPK and c["swa_window"] == oracle.SWA_W
    assert c["pool_max_blocks"] == oracle.POOL_BLOCKS and c["pool_block_positions"] == oracle.BLOCK
    assert c["max_context"] == 2 ** 20
    # encoder chunked prefill workload: (65,536 prefix + 8,192 new) tokens at m = 2
    assert (65536 + 8192) // c["compression_ratio_encoder"] == 36864


def test_entry_bytes():
    c = _json("config_table.json")
    mx = c["head_dim"] * 4 // 8 + c["head_dim"] // 32          # E2M1 nibbles + one E8M0 per 32
    ik = c["indexer_dim"] * 1 + 4                               # e4m3 + fp32 scale
    swa = c["head_dim"] * 1 + 4
    assert (mx, ik, swa, mx + ik) == (272, 132, 516, 404)
    codes, scales = oracle.quant_mxfp4(np.ones((1, 512), np.float32))
    assert codes.nbytes + scales.nbytes == 272


def test_footprint_numbers_consistent():
    f = _json("footprint.json")
    assert abs(389120 / f["ratio_vs_v1"] - f["global_kv_bytes_per_token"]) < 1.0
    assert abs(f["one_million_tokens_v4_flash_gb"] * 1000 * f["ratio_vs_v4_flash"]
               - f["one_million_tokens_global_kv_mb"]) < 1.0
    assert f["global_kv_bytes_per_token"] * 10 ** 6 / 10 ** 6 == f["one_million_tokens_global_kv_mb"]


def test_layer_grouping():
    t = _json("mode_table.json")
    dec = t["decoder_first_group"] + t["decoder_later_group"] * t["decoder_later_groups"]
    assert dec == oracle.DECODER_PATTERN and len(dec) == t["decoder_layers"]
    assert t["encoder_group"] == oracle.ENCODER_GROUP
    assert 3 * len(t["encoder_group"]) == t["encoder_csa2_layers"]
    assert t["encoder_csa2_layers"] + t["encoder_pure_swa_layers"] == 20
    assert t["modes"]["reuse"]["computes"] == []


# ---------------------------------------------------------------- generator
def test_hash_host_and_torch_agree():
    for stream, start, count in [(synth.stream_id(1, 2, 3), 0, 5000),
                                 (synth.stream_id(9), (1 << 32) - 1000, 3000),
                                 (7, 123456789, 100)]:
        a = synth.hash_np(stream, start, count)
        b = synth.hash_torch(stream, start, count, "cpu").numpy().astype(np.uint64)
        assert np.array_equal(a, b)
        assert a.max() < 2 ** 32


def test_generator_values_and_twins():
    s = synth.stream_id(5, 6)
    a = synth.normal_bf16(s, 10, 20000)
    b = synth.normal_bf16_torch(s, 10, 20000, "cpu").view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(a, b)
    assert np.array_equal(synth.uniform_f32(s, 0, 999), synth.uniform_f32_torch(s, 0, 999, "cpu").numpy())
    assert np.array_equal(synth.normal_f32(s, 0, 999, 0.1), synth.normal_f32_torch(s, 0, 999, "cpu", 0.1).numpy())
    # slices regenerate independently
    assert np.array_equal(synth.normal_bf16(s, 0, 30000)[10:20010], a)


def test_generator_distributions():
    s = synth.stream_id(77)
    x = synth.bf16_bits_to_f32(synth.normal_bf16(s, 0, 1 << 20)).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    u = synth.uniform_f32(s, 0, 1 << 20).astype(np.float64)
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 3e-3
    # table rounding agrees with torch's float32 -> bfloat16 cast
    v = synth.normal_table_f32(1.0)
    t = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.normal_table_bf16(1.0), t)
