"""Byte-accounting helpers against the numbers the pages print."""
import json
import os

from paged_kv_decode_21_gb300 import traffic
from paged_kv_decode_21_gb300.workloads import CONFIGS, draw_context_lens

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


def test_decode_step_kv_bytes_worked_example():
    g = GOLD["decode_step_kv_bytes"]
    v = traffic.decode_step_kv_bytes(g["num_layers"], g["num_kv_heads"], g["head_dim"],
                                     g["context_len"], g["elem_bytes"])
    assert v == g["value"]
    assert abs(v / 2**30 - g["stated_approx_gb"]) < 0.5


def test_m_block_worked_example():
    g = GOLD["m_block"]
    assert traffic.m_block(g["bytes_per_param"], g["head_dim"], g["block_tokens"]) == g["value"]


def test_l2_resident_batches_worked_example():
    g = GOLD["l2_resident_batches"]
    mb = traffic.m_block(2, 128, 16)
    assert traffic.l2_resident_batches(g["l2_bytes"], mb, g["n_thread"], g["num_heads"]) == g["value"]


def test_algorithmic_bytes_fixed_length_configs():
    # K+V rows plus Q and out, by hand for the two fixed-length model shapes
    c = CONFIGS["llama2_7b_mha"]
    lens = draw_context_lens(c).tolist()
    assert traffic.algorithmic_bytes(lens, 32, 32, 128) == 2 * 64 * 2048 * 32 * 128 * 2 + 2 * 64 * 32 * 128 * 2
    assert traffic.algorithmic_bytes(lens, 32, 32, 128) == 2148532224
    c = CONFIGS["qwen25_7b_gqa7"]
    lens = draw_context_lens(c).tolist()
    assert traffic.algorithmic_bytes(lens, 28, 4, 128) == 4298637312
    c = CONFIGS["tiny"]
    assert traffic.algorithmic_bytes([37, 100], 4, 4, 64) == 142336
