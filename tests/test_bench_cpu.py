"""Host bookkeeping on CPU: the bench's graph-replay plan and the FLOP
accounting that turns times into TFLOP/s, and the Python binding's shared
workspace cache."""

import pytest
import torch

import bench
import workloads


def _steps_of(plan, per, nsets):
    """Expand a replay plan into the input set of every step it enqueues."""
    out = []
    for kind, k in plan:
        out += list(range(nsets)) * (per // nsets) if kind == "block" else [k]
    return out


@pytest.mark.parametrize("steps", [0, 1, 5, 16, 17, 1000])
@pytest.mark.parametrize("per,nsets", [(16, 1), (16, 2), (15, 3), (16, 8)])
def test_replay_plan_enqueues_exactly_the_steps_in_rotation(steps, per, nsets):
    sets = _steps_of(bench.replay_plan(steps, per, nsets), per, nsets)
    assert sets == [i % nsets for i in range(steps)]


def test_replay_plan_rejects_a_block_of_partial_rotations():
    with pytest.raises(ValueError):
        bench.replay_plan(10, 16, 3)


def test_causal_flops_are_half_the_square():
    w = workloads.get("long-causal-4096")
    f = bench.fwd_flops(w)
    assert f == pytest.approx(4 * w.d * w.B * w.H * w.N * w.N / 2, rel=0.01)


def test_key_padding_flops_count_valid_keys_only():
    w = workloads.get("bert-large")
    lens = torch.full((w.B,), w.N // 2, dtype=torch.int32)
    assert bench.fwd_flops(w, key_lens=lens) == pytest.approx(
        4 * w.d * w.H * w.N * (w.N // 2) * w.B)


def test_block_sparse_flops_count_kept_blocks_only():
    w = workloads.get("block-sparse-64k")
    nb = (w.N + 127) // 128
    bm = torch.zeros((nb, nb), dtype=torch.uint8)
    bm[0, 0] = 1
    bm[3, 7] = 1
    assert bench.fwd_flops(w, block_mask=bm) == pytest.approx(
        4 * w.d * w.B * w.H * 2 * 128 * 128)


def test_cached_workspace_grows_and_keeps_what_it_replaced():
    # the binding's shared workspace (exercised on the CPU device): replaced
    # buffers stay referenced, since a captured CUDA graph may still use them
    from exact_attention_12_gb300 import api
    dev = torch.device("cpu")
    key = (dev.type, dev.index)
    api._workspaces.pop(key, None)
    api._retired.pop(key, None)
    a = api.workspace(dev, 1000)
    assert a.numel() == 1000 and not a.any()
    assert api.workspace(dev, 600) is a                 # big enough: reused
    b = api.workspace(dev, 1500)
    assert b.numel() == 2000                            # grows at least twofold
    assert len(api._retired[key]) == 1 and api._retired[key][0] is a
    c = api.workspace(dev, 10 ** 5)
    assert c.numel() == 10 ** 5
    assert [id(t) for t in api._retired[key]] == [id(a), id(b)]
    api._workspaces.pop(key, None)
    api._retired.pop(key, None)


@pytest.mark.parametrize("name,over", [("long-causal-512", {}), ("bert-large", {}),
                                       ("block-sparse-64k", {"N": 1000, "H": 2}),
                                       ("gqa-4k", {"N": 700, "B": 1})])
def test_oracle_units_cover_the_workload_and_count_its_flops(name, over):
    # the oracle's timing units (whole heads or row blocks) partition the
    # workload, and their FLOPs add up to the step's fwd+bwd FLOPs
    w = workloads.get(name, **over)
    inp = workloads.make_inputs(w)
    if w.block_density is not None:
        nb = (w.N + 127) // 128
        inp["block_mask"] = workloads.make_block_mask(nb, 0.3, seed=3)
    units = bench.oracle_units(w)
    seen = {}
    for b, h, rows in units:
        for r in rows.tolist():
            seen[(b, h, r)] = seen.get((b, h, r), 0) + 1
    assert len(seen) == w.B * w.H * w.N and set(seen.values()) == {1}
    total = sum(bench.rows_flops(w, inp, b, rows) for b, h, rows in units)
    want = 3.5 * bench.fwd_flops(w, inp["key_lens"], inp["block_mask"])
    # the metric counts causal work as N^2 / 2; the rows' exact count of
    # allowed pairs is N (N + 1) / 2
    assert total == pytest.approx(want * ((w.N + 1) / w.N if w.causal else 1.0), rel=1e-12)


def test_oracle_sample_runs_and_counts_what_it_did():
    w = workloads.get("long-causal-512", H=2)
    inp = workloads.make_inputs(w)
    units = bench.oracle_units(w)
    f, dt, n = bench.oracle_sample(w, inp, units, bench.oracle_inputs(inp), 0.0)
    assert n == 1 and dt > 0
    assert f == bench.rows_flops(w, inp, units[0][0], units[0][2])


def test_stage_bytes_of_a_plain_head():
    w = workloads.get("long-causal-4096", H=1)
    fwd, pre, main, dq = bench.stage_bytes(w)
    nd = w.N * w.d
    assert fwd == 2 * 4 * nd + 4 * w.N                 # Q, K, V read; O, L written
    assert dq == 6 * nd                                # fp32 accumulator in, bf16 dQ out
    assert main > 2 * 6 * nd and pre > 2 * 2 * nd


def _profile(tmp_path, line):
    (tmp_path / "x.md").write_text("# summary\n\n    " + line + "\n")


def test_traffic_is_read_from_profiles_while_the_sources_match(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    h = bench.kernel_source_hash("bwd_bf16_kernel")
    _profile(tmp_path, f"traffic-per-launch | bwd_bf16_kernel | long-causal-16384 | 123456 | src {h}")
    got, note = bench.profiled_traffic("bwd_bf16_kernel", "long-causal-16384")
    assert got == 123456.0 and "x.md" in note
    assert bench.profiled_traffic("bwd_bf16_kernel", "bert-large")[0] is None
    assert bench.profiled_traffic("fwd_bf16_kernel", "long-causal-16384")[0] is None


def test_traffic_of_changed_sources_is_not_reported(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    _profile(tmp_path, "traffic-per-launch | bwd_bf16_kernel | long-causal-16384 | 99 | src 0123")
    got, note = bench.profiled_traffic("bwd_bf16_kernel", "long-causal-16384")
    assert got is None and "predates" in note


def test_roofline_takes_the_longest_stage_and_the_nearer_bound():
    w = workloads.get("long-causal-16384")
    f = bench.fwd_flops(w)
    r = dict(stage_ms=[0.8, 0.05, 2.4, 0.03], fwd_flops=f, bwd_flops=2.5 * f)
    roof = bench.roofline(w, r)
    assert roof["kernel"] == "bwd_bf16_kernel" and roof["bound"] == "tensor"
    assert roof["achieved"] == pytest.approx(2.5 * f / 2.4e-3 / 1e12)
    assert roof["frac"] == pytest.approx(roof["achieved"] / bench.peaks()[0])
    # a memory-bound stage dominating
    r = dict(stage_ms=[0.01, 0.5, 0.02, 0.01], fwd_flops=f, bwd_flops=2.5 * f)
    roof = bench.roofline(w, r)
    assert roof["kernel"] == "bwd_preprocess_kernel" and roof["bound"] == "hbm"
    assert roof["unit"] == "GB/s"


def test_workload_overrides_parse_into_fields():
    assert bench.parse_overrides(["H=2", "dropout_p=0.25", "dtype=fp8"]) == \
        {"H": 2, "dropout_p": 0.25, "dtype": "fp8"}
    with pytest.raises(SystemExit):
        bench.parse_overrides(["heads=2"])
    w = workloads.get("long-causal-16384", **bench.parse_overrides(["H=2"]))
    assert (w.H, w.N, w.d, w.causal) == (2, 16384, 128, True)


def test_nvtx_ranges_need_no_profiler():
    # the bench's phases sit in NVTX ranges; entering one must work on a host
    # without a GPU or a profiler attached
    with bench.nvtx("phase"):
        with bench.nvtx("nested"):
            pass


@pytest.mark.parametrize("name", ["single-head-fp32", "fp8-long-causal-512"])
def test_forward_only_oracle_sample(name):
    # forward-only workloads are timed on the oracle head by head; at least
    # one head runs, and the FLOPs are whole heads' worth
    w = workloads.get(name)
    flops, dt, done = bench.fwd_only_oracle_sample(w, 0.0)
    assert done == 1 and dt > 0
    assert flops == bench.fwd_flops(workloads.get(name, B=1, H=1, H_kv=1))


def test_headline_line_carries_the_contract_keys():
    # the training-step line from a measurement (made up here): every key the
    # bench contract names, the roofline of the dominant stage with a traffic
    # figure read from profiles/ when it is current, and value = the whole
    # step's FLOPs over its time
    w = workloads.get("long-causal-16384")
    ff = bench.fwd_flops(w)
    r = dict(ms_per_step=3.0, stage_ms=[0.75, 0.04, 2.2, 0.03], fwd_flops=ff, bwd_flops=2.5 * ff,
             nsets=1, resident_bytes=643 << 20, launches=800,
             clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    line = bench.headline_line(w, r, steps=200, warmup=20, world=1)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "gpu_launches", "roofline", "clocks"):
        assert key in line, key
    assert line["value"] == pytest.approx(3.5 * ff / 3.0e-3 / 1e12)
    assert line["config"]["workload"].startswith("long-causal-16384")
    roof = line["roofline"]
    assert roof["kernel"] == "bwd_bf16_kernel" and roof["bound"] == "tensor"
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert set(roof) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
