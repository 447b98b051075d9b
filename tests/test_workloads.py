"""Checks on the synthetic workloads (CPU only): shapes against the pages'
KV-size figures, and structural validity of tables and slot mappings."""
import numpy as np
import pytest

import workloads as W
from tests._golden import load

KV = load("kv_size_formula.json")


def _per_token_all_layers(name, layers):
    c = W.CONFIGS[name]
    elt = 1 if c["cache_dtype"] in ("e4m3", "e5m2") else 2
    return 2 * layers * c["Hkv"] * c["d"] * elt


def test_llama2_shape_matches_page_size():
    g = KV["llama2_7b"]
    total = _per_token_all_layers("llama2-7b", g["layers"]) * g["seq_len"]
    assert abs(total - g["approx_bytes"]) / g["approx_bytes"] < 0.1


def test_opt13b_shape_matches_page_size():
    g = KV["opt13b"]
    total = _per_token_all_layers("opt13b-beam", g["layers"]) * g["seq_len"]
    assert abs(total - g["approx_bytes"]) / g["approx_bytes"] < 0.1


def test_qwen3_shape_matches_page_size():
    g = KV["qwen3_0_6b"]
    per_tok = _per_token_all_layers("qwen3-prefix", g["layers"])
    assert per_tok == g["bytes_per_token"]
    assert per_tok * g["seq_len"] == g["bytes_per_seq_mib"] * 2 ** 20


@pytest.mark.parametrize("name", W.ALL_CONFIGS)
def test_structure_is_valid(name):
    st = W.build_structure(name, 1)
    bs, nb = st["cfg"]["bs"], st["num_blocks"]
    lens, bt = st["seq_lens"], st["block_tables"]
    assert sorted(st["pool_order"].tolist()) == list(range(nb))
    for s in range(st["S"]):
        nblk = -(-int(lens[s]) // bs)
        row = bt[s, :nblk]
        assert ((row >= 0) & (row < nb)).all()
        assert len(set(row.tolist())) == nblk
    assert len(set(st["ctx_slots"].tolist())) == len(st["ctx_slots"])
    allslots = np.concatenate([st["ctx_slots"], st["new_slots"]])
    assert ((allslots >= 0) & (allslots < nb * bs)).all()
    # copy-on-write destinations are distinct and never a source
    pairs = st["cow_pairs"]
    if len(pairs):
        assert len(set(pairs[:, 1].tolist())) == len(pairs)
        assert set(pairs[:, 1].tolist()).isdisjoint(pairs[:, 0].tolist())


def test_named_sizes():
    st = W.build_structure("llama2-7b", 2)
    assert st["S"] == 64 and st["seq_lens"].min() >= 512 and st["seq_lens"].max() <= 4096
    st = W.build_structure("qwen3-prefix", 3)
    assert (st["block_tables"][:, :64] == st["block_tables"][0, :64]).all()
    st = W.build_structure("opt13b-beam", 4)
    assert st["S"] == 128
    st = W.build_structure("gqa-fp8", 5)
    assert st["seq_lens"].min() >= 256 and st["seq_lens"].max() <= 32768
