"""Pins the cost model to the numbers the pages print (tests/golden/pages_numbers.json)."""
import json
import os

import pytest

from dsa_sparse_mla_gb300 import costmodel as cm


@pytest.fixture(scope="module")
def pages(golden_dir):
    with open(os.path.join(golden_dir, "pages_numbers.json")) as f:
        return json.load(f)


def test_row_and_head_costs(pages):
    assert cm.mla_row_bytes() == pages["row_bytes"]
    assert cm.mla_head_bytes() == pages["head_bytes"]
    assert cm.mla_flops_per_row_head() == pages["flops_per_row_head"]
    assert round(pages["rows_per_query"] * cm.mla_row_bytes() / 1e6, 2) == pages["bytes_per_query_MB"]


@pytest.mark.parametrize("heads,key", [(8, "heads8"), (64, "heads64")])
def test_intensity(pages, heads, key):
    want = pages[key]
    rows = pages["rows_per_query"]
    assert round(cm.mla_query_flops(heads, rows) / 1e6, 1) == pytest.approx(want["MFLOP"], abs=0.5)
    assert round(cm.mla_query_bytes(heads, rows) / 1e6, 2) == want["MB"]
    assert round(cm.mla_intensity(heads, rows)) == want["flops_per_byte"]


def test_h200_ridge(pages):
    h = pages["h200"]
    assert round(cm.ridge(h["dense_bf16_tflops"] * 1e12, h["tb_per_s"] * 1e12)) == h["ridge_flops_per_byte"]


def test_kv_footprint(pages):
    t = pages["kv_per_token_terms"]
    assert cm.kv_bytes_per_token(t["mla_layers"], t["indexer_layers"], t["indexer_row"] - 4, t["mtp"]) == pages["kv_per_token_bytes"]
    gib = cm.kv_gib_per_request(pages["tokens_1M"])
    assert round(gib, 1) == pages["kv_1M_GiB"]
    assert round(gib / 8, 1) == pages["kv_1M_GiB_per_gpu_dcp8"]


def test_indexer_crossover(pages):
    tp8 = cm.indexer_crossover_tokens(gpus=8, shard_indexer=False)
    pcp8 = cm.indexer_crossover_tokens(gpus=8, shard_indexer=True)
    # the pages round to ~32K and ~256K
    assert abs(tp8 - pages["crossover_tokens_tp8_approx"]) / pages["crossover_tokens_tp8_approx"] < 0.03
    assert abs(pcp8 - pages["crossover_tokens_pcp8_approx"]) / pages["crossover_tokens_pcp8_approx"] < 0.03
    assert pcp8 / tp8 == pytest.approx(8.0)
