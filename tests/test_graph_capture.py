"""A training step (dlrm_sparse_fwd with pooled_save, then dlrm_sparse_bwd_adagrad,
or the split step: dlrm_sparse_bwd_sort beside the forward, then
dlrm_sparse_bwd_update_sorted) captured into a CUDA graph and replayed gives,
bitwise, what the same steps give when called directly: the caller's side
stream forks from and joins the captured stream (through events), and every
kernel of the step is deterministic.  Steps queued on independent streams at once give
the results of the same steps run one after another: the library holds no
state shared between calls."""
import numpy as np
import pytest
import torch

import embedding_bag_lookup_dlrm_b300 as dl
from gpu_util import dev_index, dev_tables, random_case

pytestmark = pytest.mark.gpu


class Step:
    """Buffers of one training step, allocated once, so that a graph can replay it."""

    def __init__(self, tabs, Vs, idx, off, dense, grad_out, D, side=None, split=False):
        B, T = dense.shape[0], len(tabs)
        self.side, self.split = side, split
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
        if self.split:  # the sort on the side stream beside the forward; the per-row sums wait for its event
            cur = torch.cuda.current_stream()
            fork, sorted_ev = torch.cuda.Event(), torch.cuda.Event()
            fork.record(cur)
            self.side.wait_event(fork)
            dl.dlrm_sparse_bwd_sort(self.tables, self.di, self.do, self.ws, status=self.status, stream=self.side)
            sorted_ev.record(self.side)
            dl.dlrm_sparse_fwd(self.tables, self.di, self.do, self.dx, out=self.out, pooled_save=self.ps,
                               status=self.status)
            dl.dlrm_sparse_bwd_update_sorted(self.tables, self.di, self.do, self.dx, self.ps, self.g, "adagrad",
                                             0.01, 1e-8, self.accum, grad_dense=self.gd, workspace=self.ws,
                                             status=self.status, sorted=sorted_ev)
            return
        dl.dlrm_sparse_fwd(self.tables, self.di, self.do, self.dx, out=self.out, pooled_save=self.ps,
                           status=self.status)
        dl.dlrm_sparse_bwd_adagrad(self.tables, self.accum, self.di, self.do, self.dx, self.ps, self.g, 0.01, 1e-8,
                                   grad_dense=self.gd, workspace=self.ws, status=self.status, side_stream=self.side)

    def state(self):
        return [t.clone() for t in self.tables] + [a.clone() for a in self.accum] + [self.out.clone(),
                                                                                      self.gd.clone()]


@pytest.mark.parametrize("layout", ["side-stream", "one-stream", "split"])
def test_graph_replay_matches_direct_calls(layout):
    """layout "split": dlrm_sparse_bwd_sort on the side stream beside the forward, then
    dlrm_sparse_bwd_update_sorted waiting for the sort's event, captured the same way."""
    B, T, D, V = 3000, 26, 128, 500
    tabs, Vs, idx, off, dense = random_case(77, B, T, D, V, 1, 8, value_scale=0.05)
    g = np.random.default_rng(5).standard_normal((B, D + (T + 1) * T // 2)).astype(np.float32)
    side = torch.cuda.Stream(priority=-100) if layout != "one-stream" else None
    split = layout == "split"

    direct = Step(tabs, Vs, idx, off, dense, g, D, side, split)
    direct.run()
    torch.cuda.synchronize()
    after_one = direct.state()
    direct.run()
    torch.cuda.synchronize()
    after_two = direct.state()

    graphed = Step(tabs, Vs, idx, off, dense, g, D, side, split)
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


@pytest.mark.parametrize("two_streams", [True, False], ids=["side-stream", "one-stream"])
def test_step_on_another_stream_matches_default_stream(two_streams):
    """The step called on a non-default stream gives the default stream's results, and work queued on
    that stream right after the call (copies of the updated state, no synchronisation in between)
    already sees them: the side stream joins the caller's stream before the call returns."""
    B, T, D, V = 2000, 26, 128, 300
    tabs, Vs, idx, off, dense = random_case(78, B, T, D, V, 1, 8, value_scale=0.05)
    g = np.random.default_rng(6).standard_normal((B, D + (T + 1) * T // 2)).astype(np.float32)
    ref = Step(tabs, Vs, idx, off, dense, g, D)
    ref.run()
    torch.cuda.synchronize()
    expected = ref.state()

    step = Step(tabs, Vs, idx, off, dense, g, D, torch.cuda.Stream() if two_streams else None)
    other = torch.cuda.Stream()
    other.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(other):
        step.run()
        snap = step.state()
    torch.cuda.synchronize()
    for a, b in zip(snap, expected):
        assert torch.equal(a, b)


def test_independent_streams_run_at_once():
    """Two steps on their own tables, queued together on two streams (each with its own side stream),
    give what each gives alone."""
    B, T, D, V = 2500, 26, 128, 400
    cases = []
    for k in range(2):
        tabs, Vs, idx, off, dense = random_case(90 + k, B, T, D, V, 1, 8, value_scale=0.05)
        g = np.random.default_rng(20 + k).standard_normal((B, D + (T + 1) * T // 2)).astype(np.float32)
        cases.append((tabs, Vs, idx, off, dense, g))
    expected = []
    for c in cases:
        alone = Step(*c, D)
        alone.run()
        torch.cuda.synchronize()
        expected.append(alone.state())
    steps = [Step(*c, D, torch.cuda.Stream()) for c in cases]
    streams = [torch.cuda.Stream() for _ in cases]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for step, st in zip(steps, streams):
        with torch.cuda.stream(st):
            step.run()
    torch.cuda.synchronize()
    for step, exp in zip(steps, expected):
        for a, b in zip(step.state(), exp):
            assert torch.equal(a, b)
