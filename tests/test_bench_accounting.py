"""The bench's algorithmic work, counted here a second way: prefill FLOPs from the (row, key)
pairs that causal chunked attention lets through, decode bytes from the cache slots and
block-table entries each sequence's keys occupy; and the rule that ties committed ncu
traffic to the kernel sources it was taken on."""
import json

import pytest
import torch

import bench
import workloads


def _visible_pairs(case):
    """Rows of each chunk at absolute positions C - Lq .. C - 1 see keys 0 .. position."""
    qsl = case.query_start_loc.tolist()
    n = 0
    for s in range(case.num_seqs):
        lq, c = qsl[s + 1] - qsl[s], int(case.context_lens[s])
        for row in range(lq):
            pos = c - lq + row
            n += sum(1 for key in range(c) if key <= pos)
    return n


@pytest.mark.parametrize("prefixes,chunks", [([0, 5, 17], [3, 4, 2]), ([0], [1]), ([40, 0], [9, 13])])
def test_prefill_flops_count_the_visible_pairs(prefixes, chunks):
    case = workloads.make_prefill_case("acct", prefixes, chunks, 8, 4, 2, 64, torch.bfloat16, 3)
    flops, byts = bench.prefill_work(case)
    # two products per visible (row, key): q.k over D and p.v over D, 2 flops per multiply-add
    assert flops == 2 * 2 * case.head_dim * case.num_heads * _visible_pairs(case)
    kv = sum(int(c) for c in case.context_lens) * case.num_kv_heads * case.head_dim * 2 * 2
    assert byts == kv + case.query.numel() * 2 + case.query.numel() * 4


def test_decode_bytes_count_the_slots_and_table_entries_read():
    case = workloads.make_decode_case("acct", [1, 7, 8, 9, 33, 100], 8, 8, 2, 64, torch.float16, 4,
                                      free_frac=0.2)
    b = bench.decode_bytes(case)
    row = case.num_kv_heads * case.head_dim * 2      # one token of one sequence, fp16
    slots, entries = 0, 0
    for s in range(case.num_seqs):
        c = int(case.context_lens[s])
        bt = case.block_tables[s].tolist()
        seen = {(bt[t // case.block_size], t % case.block_size) for t in range(c)}
        slots += len(seen)
        entries += len({t // case.block_size for t in range(c)})
    assert b["kv"] == slots * row * 2                # K and V
    q = case.num_seqs * case.num_heads * case.head_dim
    assert b["decode"] == b["kv"] + q * 2 + q * 4 + entries * 4 + case.num_seqs * 4
    fresh = case.num_seqs * row * 2 * 2 + case.num_seqs * 8
    assert b["step"] == b["decode"] + fresh


def test_kernel_hash_ignores_comments_only():
    code = "int f(int x) {\n    return x + 1;  // add\n}\n/* note\n spanning lines */\n"
    same = "// header\nint f(int x) {\n\n    return x + 1;\n}\n"
    other = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)


def test_traffic_is_reported_only_for_the_sources_it_was_taken_on(monkeypatch, tmp_path):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(
        {"decode": {"long_decode": {"source_sha256_16": "abc", "dram_bytes_per_launch": 123}}}))
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kind="decode": "abc")
    assert bench.profiled_traffic("decode", "long_decode") == 123
    assert bench.profiled_traffic("decode", "decode_batch") is None
    assert bench.profiled_traffic("prefill", "prefill_chunk") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kind="decode": "changed")
    assert bench.profiled_traffic("decode", "long_decode") is None
