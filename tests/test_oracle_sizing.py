"""Pins for the oracle's sizing arithmetic against the numbers the pages print.

Fixtures: tests/golden/kv_size_examples.json (each entry cites its page and
section).  A dropped factor (K/V, bytes, layers, batch) moves every result
by at least 2x and fails here.
"""
import json
import os

import pytest

from oracle import sizing
from oracle.allocator import AllocatorModel

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "kv_size_examples.json")))
UNIT = {"MB": 1e6, "GB": 1e9, "MiB": 2 ** 20, "GiB": 2 ** 30, "elements": 1}


def evaluate(form, i):
    if form == "hidden":
        return sizing.kv_bytes_from_hidden(i["layers"], i["seq_len"], i["hidden"], i["batch"], i["bytes"])
    if form == "general":
        return sizing.kv_bytes(i["layers"], i["kv_heads"], i["head_dim"], i["seq_len"], i["batch"], i["bytes"])
    if form == "layer_elements":
        return sizing.layer_kv_elements(i["batch"], i["seq_len"], i["kv_heads"], i["head_dim"])
    if form == "request_bound":
        return sizing.request_kv_bound(i["max_seq_len"], i["layers"], i["kv_heads"], i["head_dim"], i["bytes"])
    raise KeyError(form)


@pytest.mark.parametrize("ex", GOLDEN["examples"], ids=lambda e: e["id"])
def test_printed_examples(ex):
    value = evaluate(ex["form"], ex["inputs"]) / UNIT[ex["unit"]]
    if ex["tol"] == 0:
        assert value == ex["printed"]
    else:
        assert abs(value - ex["printed"]) <= ex["tol"]


def test_hidden_and_general_forms_agree_for_mha():
    # kv_heads * head_dim == hidden for multi-head attention
    assert sizing.kv_bytes_from_hidden(40, 2048, 4096, 8) == sizing.kv_bytes(40, 32, 128, 2048, 8, 2)


@pytest.mark.parametrize("cap", GOLDEN["capacity"], ids=lambda c: c["id"])
def test_capacity_examples(cap):
    gb = 1e9 if cap["per_request"].get("unit", "GB") == "GB" else 2 ** 30
    budget = sizing.kv_budget(cap["memory_gb"] * gb, cap["utilisation"], cap["weights_gb"] * gb)
    assert budget / gb == pytest.approx(cap["printed_budget_gb"], abs=1e-9)
    if "printed_usable_gb" in cap:
        assert cap["memory_gb"] * cap["utilisation"] == pytest.approx(cap["printed_usable_gb"])
    per = evaluate(cap["per_request"]["form"], cap["per_request"]["inputs"])
    assert abs(per / gb - cap["printed_per_request_gb"]) <= cap["per_request_tol"]
    assert abs(sizing.max_concurrency(budget, per) - cap["printed_concurrency"]) <= cap["concurrency_tol"]


def test_fp8_halves_the_cache():
    i = GOLDEN["fp8_halves"]["inputs"]
    b16 = sizing.kv_bytes(i["layers"], i["kv_heads"], i["head_dim"], i["seq_len"], i["batch"], 2)
    b8 = sizing.kv_bytes(i["layers"], i["kv_heads"], i["head_dim"], i["seq_len"], i["batch"], 1)
    assert b8 * 2 == b16
    # with one fp32 scale per (token, KV head) the overhead is 4 / head_dim
    per_tok = sizing.fp8_bytes_per_token(i["layers"], i["kv_heads"], i["head_dim"])
    assert per_tok * i["seq_len"] == b8 * (1 + 4 / i["head_dim"])


def test_allocated_bytes_match_closed_form():
    # a paged allocation of L tokens holds ceil(L/16)*16 slots; at multiples of 16 it equals the formula
    layers, hkv, d = 32, 8, 128
    per_block = sizing.kv_bytes(layers, hkv, d, 16, 1, 2)
    for lens in ([32768], [1, 16, 17, 100], [2048] * 8):
        a = AllocatorModel(sum(-(-L // 16) for L in lens) + 3)
        for s, L in enumerate(lens):
            a.create(s)
            a.append_slots([s] * L)
        held = (a.num_blocks - a.num_free()) * per_block
        assert held == sizing.kv_bytes(layers, hkv, d, sizing.paged_token_slots(lens), 1, 2)
        if all(L % 16 == 0 for L in lens):
            assert held == sum(sizing.kv_bytes(layers, hkv, d, L, 1, 2) for L in lens)
    assert sizing.kv_bytes(32, 8, 128, 32768, 1, 2) == 4 * 2 ** 30


def test_utilisation_and_pool_sizing():
    lens = [1, 16, 17, 100]
    assert sizing.paged_utilisation(lens) == 134 / (16 + 16 + 32 + 112)
    assert sizing.prealloc_utilisation(lens, 2048) == 134 / (4 * 2048)
    per_block = 2 * 40 * 32 * 16 * 128 * 2
    assert sizing.pool_blocks(10 * per_block + 5, 40, 32, 128, "f16") == 10
    assert sizing.pool_blocks(2 * 1 * 8 * 16 * 132 * 3, 1, 8, 128, "fp8_e4m3") == 3
