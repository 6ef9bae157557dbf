"""Host-side logic of bench.py on CPU: multi-rank timing over gloo, byte accounting,
clock-sample parsing and the peak fallback (no GPU)."""

import os
import socket
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own duration; the job takes the slowest
        got = bench.max_over_ranks(0.5 + rank, dist, torch.device("cpu"))
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world_size_2_gloo():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 1.5, 1: 1.5}


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(0.25, None, None) == 0.25


def test_rank_seeds_differ_per_rank_and_set():
    seeds = {bench.rank_seed(1001, r, b) for r in range(8) for b in range(3)}
    assert len(seeds) == 24


def test_verify_bytes_single_user_launch():
    # 48 layers x 48 heads: state 32 KiB + 16 x (q,k,v,o 4 x 256 B) + 16 x 8 B + 16 x 32 KiB
    per_head = 32768 + 16 * 1024 + 128 + 16 * 32768
    assert bench.verify_bytes(48, 16, 48, 128, 128, 2) == 48 * 48 * per_head == 1321500672


def test_commit_and_accept_bytes():
    acc = torch.tensor([15])
    assert bench.commit_bytes(48, acc, 48, 128, 128, 2) == 2 * 48 * 48 * 128 * 128 * 2
    assert bench.commit_bytes(48, torch.tensor([0]), 48, 128, 128, 2) == 0
    assert bench.accept_bytes(1, 16, 151936, 2) == 16 * 151936 * 2 + 16 * 8 + 4


def test_prefill_bytes_25k():
    # q, k, v, o + beta, g per token-head, state in + out, one checkpoint per 64 tokens
    b = bench.prefill_bytes(1, 25000, 48, 128, 128, 2)
    per_head = 25000 * (4 * 256 + 8) + 2 * 32768 + 390 * 32768
    assert b == 48 * per_head


def test_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6696.2}')
    assert bench.peaks() == (6696.2, "measured")


def test_clock_sampler_summary_parsing():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    t0 = time.time()
    stamp = lambda dt: time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t0 + dt)) + ".100"
    cs.lines = [
        "%s, 0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active" % stamp(0),
        "%s, 0, 1980, 2070, 1300.5, 0x4, Not Active, Not Active, Not Active, Active" % stamp(1),
        "%s, 1, 345, 2070, 90.0, 0x0, Not Active, Not Active, Not Active, Not Active" % stamp(1),
    ]
    s = cs.summary(t0 - 1, t0 + 2, 0)
    assert s["sm_mhz"] == pytest.approx((2070 + 1980) / 2)
    assert s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def test_kernel_sources_hash_is_stable():
    assert bench.kernel_sources_hash() == bench.kernel_sources_hash()


def test_context_bytes():
    # every token once, plus length in and (drafts, count, match length) out per request
    assert bench.context_bytes([26000], 8) == 26000 * 4 + 4 * (1 + 8 + 2)
    assert bench.context_bytes([10, 0], 4) == 40 + 2 * 4 * 7


def test_e2e_group_bounds():
    # the end-to-end step's layer groups: equal counts or explicit growing sizes
    assert bench.e2e_group_bounds(48, 1) == [0, 48]
    assert bench.e2e_group_bounds(48, 4) == [0, 12, 24, 36, 48]
    assert bench.e2e_group_bounds(48, (8, 16, 24)) == [0, 8, 24, 48]
    for bad in (5, 0, (8, 16), (8, 16, 25), (0, 24, 24)):
        with pytest.raises(ValueError):
            bench.e2e_group_bounds(48, bad)


def test_e2e_growing_groups_cover_the_layers():
    assert bench.e2e_growing_groups(48) == [4, 8, 16, 20]
    for L in (1, 5, 11, 12, 13, 47, 48, 96):
        g = bench.e2e_growing_groups(L)
        assert sum(g) == L and min(g) >= 1
        assert bench.e2e_group_bounds(L, g)[-1] == L


def test_prefill_fractions_against_both_peaks():
    row = {"per_layer_launches": {"achieved_gbs": 2000.0}, "folded_one_launch": {"achieved_gbs": 4400.0}}
    bench.add_prefill_fractions(row, 6775.9)
    assert abs(row["folded_one_launch"]["frac"] - 4400.0 / 6775.9) < 1e-12
    assert abs(row["folded_one_launch"]["frac_of_nominal_8tbs"] - 0.55) < 1e-12
    assert abs(row["per_layer_launches"]["frac"] - 2000.0 / 6775.9) < 1e-12
