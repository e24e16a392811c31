"""A training step (dlrm_sparse_fwd with pooled_save, then dlrm_sparse_bwd_adagrad)
captured into a CUDA graph and replayed gives, bitwise, what the same steps give
when called directly: the backward's side stream forks from and joins the
captured stream, and every kernel of the step is deterministic."""
import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl
from gpu_util import dev_index, dev_tables, random_case

pytestmark = pytest.mark.gpu


class Step:
    """Buffers of one training step, allocated once, so that a graph can replay it."""

    def __init__(self, tabs, Vs, idx, off, dense, grad_out, D):
        B, T = dense.shape[0], len(tabs)
        self.tables = dev_tables(tabs, "f32")
        self.accum = [torch.full((v,), 0.1, device="cuda") for v in Vs]
        self.di, self.do = dev_index(idx, "i32"), dev_index(off, "i32")
        self.dx = torch.from_numpy(dense).cuda()
        self.g = torch.from_numpy(grad_out).cuda()
        self.out = torch.empty((B, D + (T + 1) * T // 2), device="cuda")
        self.ps = torch.empty((B, T, D), device="cuda")
        self.gd = torch.empty((B, D), device="cuda")
        need = dl.dlrm_sparse_bwd_workspace_size(self.tables, self.di, self.do)
        self.ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self):
        dl.dlrm_sparse_fwd(self.tables, self.di, self.do, self.dx, out=self.out, pooled_save=self.ps,
                           status=self.status)
        dl.dlrm_sparse_bwd_adagrad(self.tables, self.accum, self.di, self.do, self.dx, self.ps, self.g, 0.01, 1e-8,
                                   grad_dense=self.gd, workspace=self.ws, status=self.status)

    def state(self):
        return [t.clone() for t in self.tables] + [a.clone() for a in self.accum] + [self.out.clone(),
                                                                                      self.gd.clone()]


def test_graph_replay_matches_direct_calls():
    B, T, D, V = 3000, 26, 128, 500
    tabs, Vs, idx, off, dense = random_case(77, B, T, D, V, 1, 8, value_scale=0.05)
    g = np.random.default_rng(5).standard_normal((B, D + (T + 1) * T // 2)).astype(np.float32)

    direct = Step(tabs, Vs, idx, off, dense, g, D)
    direct.run()  # also the first call on the device: creates the library's side stream, configures kernels
    torch.cuda.synchronize()
    after_one = direct.state()
    direct.run()
    torch.cuda.synchronize()
    after_two = direct.state()

    graphed = Step(tabs, Vs, idx, off, dense, g, D)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        graphed.run()
    # capture records and runs nothing: the tables are still the initial ones
    torch.cuda.synchronize()
    assert np.array_equal(graphed.tables[0].cpu().numpy(), tabs[0])

    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(graphed.state(), after_one):
        assert torch.equal(a, b)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(graphed.state(), after_two):
        assert torch.equal(a, b)
    assert direct.status.item() == 0 and graphed.status.item() == 0


def test_step_on_another_stream_matches_default_stream():
    """The step called on a non-default stream gives the default stream's results, and work queued on
    that stream right after the call (copies of the updated state, no synchronisation in between)
    already sees them: the library's side stream joins the caller's stream before the call returns."""
    B, T, D, V = 2000, 26, 128, 300
    tabs, Vs, idx, off, dense = random_case(78, B, T, D, V, 1, 8, value_scale=0.05)
    g = np.random.default_rng(6).standard_normal((B, D + (T + 1) * T // 2)).astype(np.float32)
    ref = Step(tabs, Vs, idx, off, dense, g, D)
    ref.run()
    torch.cuda.synchronize()
    expected = ref.state()

    step = Step(tabs, Vs, idx, off, dense, g, D)
    other = torch.cuda.Stream()
    other.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(other):
        step.run()
        snap = step.state()
    torch.cuda.synchronize()
    for a, b in zip(snap, expected):
        assert torch.equal(a, b)
