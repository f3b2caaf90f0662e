"""Host-side models of bench.py (CPU): the per-step algorithmic bytes against the sizes the
pages print, and the agent-replay turn plan."""
import json
import os

import pytest

pytest.importorskip("torch")
import bench  # noqa: E402
import synth  # noqa: E402

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "e2b_printed_sizes.json")))


def test_weight_bytes_match_printed_checkpoint_sizes():
    """A step streams every linear and the tied lm_head once; the checkpoint the pages print
    also holds the per-layer table (gathered, not streamed) and the norm gains (< 1 MB)."""
    cfg = synth.get_config("e2b")
    table = cfg["vocab"] * cfg["num_layers"] * cfg["ple_dim"] * 2
    w_bf16, _ = bench.algorithmic_bytes(cfg, "bf16", 1, [0])
    assert abs(w_bf16 - (GOLDEN["bf16_weight_bytes"]["value"] - table)) < 1e6
    w_w4, _ = bench.algorithmic_bytes(cfg, "w4a16", 1, [0])
    assert abs(w_w4 - (GOLDEN["w4a16_weight_gb"]["value"] * 1e9 - table)) < 2e6  # 3 printed decimals


def test_kv_bytes_per_step_at_context_639():
    """12 sliding owning layers read min(T, 512) keys of 1 KB (K and V, d = 256), 3 full ones
    T keys of 2 KB; plus the new K/V row (18,432 B), the per-layer-embedding row and the
    embedding row: ~10.2 MB per sequence at T = 639."""
    cfg = synth.get_config("e2b")
    _, kv = bench.algorithmic_bytes(cfg, "w4a16", 1, [638])
    assert kv == 12 * 512 * 1024 + 3 * 639 * 2048 + GOLDEN["kv_bytes_per_token"]["value"] + 35 * 256 * 2 + 1536 * 2
    _, kv64 = bench.algorithmic_bytes(cfg, "w4a16", 64, [638])
    assert kv64 == 64 * kv


def test_replay_schedule_grows_500_to_8000_in_20_turns():
    sched = synth.replay_schedule()
    assert sched[0] == (500, 0) and len(sched) == 21
    assert all(t == (375, 32) for t in sched[1:])
    assert sched[0][0] + sum(a for a, _ in sched[1:]) == 8000
    # bench.py's replay: each turn after the first re-feeds the previous turn's last output,
    # then appends the fresh ids, then runs 31 decode steps
    ctx = sched[0][0]
    for i, (fresh, outs) in enumerate(sched[1:]):
        ctx += fresh + (1 if i > 0 else 0) + (outs - 1)
    assert ctx == 8639


def test_aliased_variant_adds_the_sharing_layers_reads():
    """Counting re-reads: the 20 KV-sharing layers (16 sliding reading layer 13, 4 full reading
    layer 14) read their source's visible keys again, and write no K/V row."""
    cfg = synth.get_config("e2b")
    _, kv = bench.algorithmic_bytes(cfg, "w4a16", 1, [638])
    _, kva = bench.algorithmic_bytes(cfg, "w4a16", 1, [638], count_aliased=True)
    assert kva - kv == 16 * 512 * 1024 + 4 * 639 * 2048
    _, kva2 = bench.algorithmic_bytes(cfg, "w4a16", 1, [99])
    _, kva3 = bench.algorithmic_bytes(cfg, "w4a16", 1, [99], count_aliased=True)
    assert kva3 - kva2 == 16 * 100 * 1024 + 4 * 100 * 2048
