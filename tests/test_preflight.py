"""The library's sizing utility against the numbers the article prints.

Article "Running an MoE Model Larger Than Your VRAM", section "A preflight script before
you turn it on": three configurations and the script's three result lines each
(tests/golden/preflight_printed.json, with its citation). The utility is a separate
implementation from the oracle's; both are pinned to the same printed values.
"""

import json
import os

import pytest

from paged_expert_moe_gb300 import preflight as pf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "preflight_printed.json")


def _cases():
    g = json.load(open(GOLDEN))
    return [(g["kv_bytes_per_token"], c) for c in g["cases"]]


@pytest.mark.parametrize("kv,case", _cases(), ids=lambda v: v["name"] if isinstance(v, dict) else str(v))
def test_sizing_reproduces_the_printed_preflight_lines(kv, case):
    s = pf.size(128, 8, 48, case["K"], expert_mb=case["expert_mb"], link_gbps=case["link_gbps"],
                tok_s=case["tok_s"], kv_bytes_per_token=kv)
    pr = case["printed"]
    assert round(s.slot_cost_mb) == pr["slot_mb"]
    assert round(s.kv_tokens_per_slot) == pr["kv_tokens"]
    assert s.batch_cap == pr["batch_cap"]
    assert round(100 * s.random_miss) == pr["random_miss_pct"]
    assert round(100 * s.max_miss) == pr["max_miss_pct"]
    assert s.reuse_implied == pr["reuse_implied"]
    lines = pf.report(s)
    assert len(lines) == 3 and ("reuse implied" in lines[2]) == pr["reuse_implied"]


def test_kv_bytes_per_token_of_the_article():
    # section "What does a resident slot cost in context length?": 2 x 48 x 4 x 128 x 2
    assert pf.qwen3_kv_bytes_per_token() == 98304


def test_sizing_from_the_library_layout():
    pytest.importorskip("ctypes")
    from paged_expert_moe_gb300 import _lib
    try:
        _lib.load()
    except Exception as e:  # the library is built by __graft_entry__.build()
        pytest.skip(f"library not built: {e}")
    # the Qwen3-30B-A3B expert in the library's three layouts
    bf = pf.size(128, 8, 48, 40, "bf16", 2048, 768)
    fp8 = pf.size(128, 8, 48, 40, "fp8", 2048, 768)
    i4 = pf.size(128, 8, 48, 26, "int4", 2048, 768, hbm_budget_gb=8.0)
    assert bf.expert_bytes == 3 * 2048 * 768 * 2 == 9_437_184
    # FP8: e4m3 codes + fp32 scales per 128x128 block; int4: packed nibbles + (s, z) fp16
    # pairs per output row and group of 128 inputs
    assert fp8.expert_bytes == 4_718_592 + 4 * 12 * 16 + 4 * 16 * 6 == 4_719_744
    assert i4.expert_bytes == 2_359_296 + 4 * 1536 * 16 + 4 * 2048 * 6 == 2_506_752
    assert i4.slot_stride % 4096 == 0 and i4.slot_stride >= i4.expert_bytes
    assert i4.arena_bytes == 26 * i4.slot_stride * 48 and i4.host_store_bytes == 128 * i4.slot_stride * 48
    assert i4.slots_fit == min(128, int(8e9 // (i4.slot_stride * 48)))
    assert bf.batch_cap == 5 and i4.batch_cap == 3
    # MXFP4: packed E2M1 codes + one E8M0 byte per output row and block of 32 inputs
    mx = pf.size(128, 8, 48, 26, "mxfp4", 2048, 768)
    assert mx.expert_bytes == 2_359_296 + 1536 * 64 + 2048 * 24 == 2_506_752


def test_cli_prints_the_three_lines(capsys):
    pf.main(["--slots", "26", "--expert-mb", "2.43", "--link-gbps", "15.75", "--tok-s", "32.6"])
    out = capsys.readouterr().out.splitlines()
    assert out[0].startswith("slot cost: 117 MB") and "1187 KV tokens" in out[0]
    assert out[1].endswith("= 3") and "reuse implied" in out[2]
