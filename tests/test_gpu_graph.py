"""A whole step captured into a CUDA graph and replayed gives exactly the
eager step's results: no call synchronises, allocates or reads host state
during the step, and every kernel's launch (with programmatic dependent
launch) is capturable."""
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


def _snapshot(w):
    out = [w.acc, w.path, w.out_tok, w.tree["parent"], w.tree["token"], w.tree["count"]]
    out += [w.flat[k] for k in ("token", "parent_row", "mask", "position", "n_rows")]
    out += [w.attn_out, w.g, w.amax, w.race_ids, w.row_max]
    return [t.clone() for t in out]


@pytest.mark.parametrize("name", ["llama8b", "serve64"])
def test_step_replays_from_a_cuda_graph(name):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = bench.Workload(name, "cuda")
    for _ in range(2):
        w.step()
    torch.cuda.synchronize()
    eager = _snapshot(w)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        w.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        w.step()
    for t in (w.acc, w.path, w.out_tok):
        t.fill_(-7)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, _snapshot(w)):
        assert torch.equal(a, b)
    assert int(w.status.item()) == 0
