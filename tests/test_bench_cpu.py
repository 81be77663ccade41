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
