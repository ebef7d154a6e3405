"""Argument checks of the Python binding that run before any launch, on CPU
tensors: caller-supplied results must match the shape, dtype, placement and
layout the kernels write, the workspace must sit on the call's device, and
the graph and parameters must sit on the device of the call."""
import types

import pytest
import torch

import graph_sparse_head_gb300 as pmha

CPU = torch.device("cpu")


def test_dest_accepts_the_exact_tensor():
    pmha._check_dest("out", torch.empty(2, 5, 8), (2, 5, 8), torch.float32, CPU)


@pytest.mark.parametrize("bad", [
    torch.empty(2, 5, 7),                           # too small
    torch.empty(2, 5, 9),                           # too large: still not the layout written
    torch.empty(2, 5, 8, dtype=torch.bfloat16),     # wrong dtype
    torch.empty(2, 8, 5).transpose(1, 2),           # strided
    "not a tensor",
])
def test_dest_refuses_other_tensors(bad):
    with pytest.raises(ValueError):
        pmha._check_dest("out", bad, (2, 5, 8), torch.float32, CPU)


def test_dest_host_only_when_asked():
    pmha._check_dest("weights", torch.empty(3, 4), (3, 4), torch.float32, None)
    meta = torch.empty(3, 4, device="meta")
    with pytest.raises(ValueError):
        pmha._check_dest("weights", meta, (3, 4), torch.float32, CPU)  # another device


def test_workspace_checks():
    ws = torch.empty(64, dtype=torch.uint8)
    assert pmha._workspace(64, CPU, ws) is ws
    with pytest.raises(ValueError):
        pmha._workspace(65, CPU, ws)  # too small
    with pytest.raises(ValueError):
        pmha._workspace(8, CPU, torch.empty(64, dtype=torch.uint8)[::2])  # strided
    with pytest.raises(ValueError):
        pmha._workspace(8, CPU, torch.empty(64, dtype=torch.uint8, device="meta"))  # elsewhere


def test_placement():
    E = 8
    t = lambda *s: torch.empty(*s)  # noqa: E731
    params = pmha.Params(t(E, E), t(E, E), t(E, E), t(E, E), t(E), None, t(E), t(E), 2)
    graph = types.SimpleNamespace(device=CPU)
    pmha._check_placement(graph, params, CPU)
    with pytest.raises(ValueError):
        pmha._check_placement(types.SimpleNamespace(device=torch.device("meta")), params, CPU)
    params.bo = torch.empty(E, device="meta")
    with pytest.raises(ValueError):
        pmha._check_placement(graph, params, CPU)
