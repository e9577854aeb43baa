"""Every entry point under CUDA graph capture: replays of a captured graph
give the eager results bit for bit. test_first_calls_inside_capture repeats
the captures in a fresh process, so that each op's first call (plan
selection, occupancy queries, shared-memory attributes, module loading)
happens inside the capture."""
import os
import subprocess
import sys

import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _capture_and_compare(run, outputs):
    """Capture run() into a graph, replay it twice, compare with an eager run."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    for o in outputs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    got = [o.clone() for o in outputs]
    for o in outputs:
        o.zero_()
    run()
    torch.cuda.synchronize()
    for a, b in zip(got, outputs):
        assert torch.equal(a, b)
    assert fn.fnorm_get_last_error() == fn.Status.OK


def test_graph_instancenorm_paths():
    ys = []
    runs = []
    for S, dt in ((256, torch.float32), (4096, torch.bfloat16), (262144, torch.float32),
                  (1000, torch.float32)):
        x = inputs.normal((3, 8, S), 5 + S, dev()).to(dt)
        y = torch.empty_like(x)
        g, b = inputs.channel_affine(8, S, dev())
        ys.append(y)
        runs.append((x, y, g, b, S, dt))

    def run():
        for x, y, g, b, S, dt in runs:
            c = fn.FNORM_F32 if dt == torch.float32 else fn.FNORM_BF16
            fn.fnorm_instancenorm_affine(x, y, g, b, 3, 8, S, c, c, EPS, None, None,
                                         torch.cuda.current_stream())
    _capture_and_compare(run, ys)


def test_graph_epilogue():
    x, m = inputs.epilogue(dev(), shape=(4, 16, 14, 30, 30))
    y = torch.empty((4, 14 * 30 * 30), device=dev())
    a = torch.empty((4, 14 * 30 * 30), dtype=torch.int64, device=dev())

    def run():
        fn.fnorm_instancenorm_epilogue(x, m, y, a, 4, 16, 14 * 30 * 30, EPS, -1.0, 1.0,
                                       torch.cuda.current_stream())
    _capture_and_compare(run, [y, a])


def test_graph_batchnorm_train_and_eval():
    x, g, b, rm, rv = inputs.batchnorm(dev(), shape=(8, 16, 63, 63))
    N, C, S = 8, 16, 63 * 63
    y = torch.empty_like(x)
    ye = torch.empty_like(x)
    ws = torch.empty(fn.fnorm_batchnorm_workspace_size(N, C, S), dtype=torch.uint8, device=dev())
    sm, sr = torch.empty(C, device=dev()), torch.empty(C, device=dev())
    rm0, rv0 = rm.clone(), rv.clone()

    def run():
        # running statistics reset inside the graph so every replay starts alike
        rm.copy_(rm0)
        rv.copy_(rv0)
        st = torch.cuda.current_stream()
        fn.fnorm_batchnorm_train(x, y, g, b, 2.0, rm, rv, 0.1, EPS, sm, sr, N, C, S, ws,
                                 ws.numel(), st)
        fn.fnorm_batchnorm_eval(x, ye, g, b, 2.0, rm, rv, EPS, N, C, S, st)
    _capture_and_compare(run, [y, ye, sm, sr, rm, rv])


def test_graph_batchnorm_resident(fnorm_env):
    """The single cooperative BatchNorm launch (with its counter reset) in a graph."""
    fnorm_env.setenv("FNORM_BN_RESIDENT", "1")
    test_graph_batchnorm_train_and_eval()


def test_first_calls_inside_capture():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("from tests import test_gpu_graphs as t; t.test_graph_instancenorm_paths(); "
            "t.test_graph_epilogue(); t.test_graph_batchnorm_train_and_eval(); print('fresh ok')")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "fresh ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]


def test_graph_instancenorm_workspace_route():
    """fnorm_instancenorm_ws on a shape that takes its workspace route (two
    BatchNorm-kernel launches on the caller's stream) and on one that does not."""
    ys, runs = [], []
    for shape in ((1, 2, 1 << 20), (2, 3, 4096)):
        N, C, S = shape
        x = inputs.normal(shape, 17 + C, dev())
        y = torch.empty_like(x)
        nb = fn.fnorm_instancenorm_workspace_size(N, C, S)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev())
        ys.append(y)
        runs.append((x, y, ws, nb, N, C, S))

    def run():
        for x, y, ws, nb, N, C, S in runs:
            fn.fnorm_instancenorm_ws(x, y, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None,
                                     ws, nb, torch.cuda.current_stream())
    _capture_and_compare(run, ys)


def test_graph_instancenorm_output_scratch_route():
    """fnorm_instancenorm without a workspace on few long fp32 slices (three
    launches that keep the per-unit statistics in the output buffer) under
    graph capture: replays equal an eager call."""
    N, C, S = 1, 2, 1 << 20
    x = inputs.normal((N, C, S), 23, dev())
    y = torch.empty_like(x)

    def run():
        fn.fnorm_instancenorm(x, y, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None,
                              torch.cuda.current_stream())
    _capture_and_compare(run, [y])
