"""The library's calls can be captured into a CUDA graph: every entry point
enqueues its kernels on the caller's stream and allocates nothing, and the
programmatic-dependent launches become graph edges.  One capture of every
operator's forward and backward, replayed, gives the same bits as the same
calls made eagerly, and replays again after the inputs change in place."""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def wsf():
    import __graft_entry__
    __graft_entry__.build()
    import backward_ws_fwd_gb300 as m
    return m


def _tensors():
    g = torch.Generator(device=DEV).manual_seed(0)
    t = {}
    t["x"] = torch.randn(4096, 1000, device=DEV, generator=g).bfloat16()
    t["w"] = torch.randn(1000, device=DEV, generator=g) * 0.03
    t["dyv"] = torch.randn(4096, device=DEV, generator=g).bfloat16()
    t["xs"] = (torch.randn(1 << 20, device=DEV, generator=g) * 2).half()
    t["dys"] = torch.randn(1 << 20, device=DEV, generator=g).half()
    t["ws"] = torch.tensor([0.75], device=DEV)
    t["dyn"] = torch.randn(4096, 1000, device=DEV, generator=g).bfloat16()
    t["wn"] = 1 + 0.1 * torch.randn(1000, device=DEV, generator=g)
    t["bn"] = 0.1 * torch.randn(1000, device=DEV, generator=g)
    return t


def _outputs(wsf, t):
    o = {}
    o["y"] = torch.empty(4096, dtype=torch.bfloat16, device=DEV)
    o["dx"] = torch.empty_like(t["x"])
    o["gw"] = torch.empty(1000, device=DEV)
    o["ws_ws"] = torch.empty(wsf.ws_bwd_workspace_bytes(4096, 1000, torch.bfloat16), dtype=torch.uint8,
                             device=DEV)
    o["ys"] = torch.empty_like(t["xs"])
    o["dxs"] = torch.empty_like(t["xs"])
    o["dws"] = torch.empty(1, device=DEV)
    o["silu_ws"] = torch.empty(wsf.silu_bwd_workspace_bytes(1 << 20, torch.float16), dtype=torch.uint8,
                               device=DEV)
    o["ym"] = torch.empty_like(t["x"])
    o["dxm"] = torch.empty_like(t["x"])
    o["yn"] = torch.empty_like(t["x"])
    o["dxn"] = torch.empty_like(t["x"])
    o["gwn"] = torch.empty(1000, device=DEV)
    o["gbn"] = torch.empty(1000, device=DEV)
    o["norm_ws"] = torch.empty(wsf.norm_bwd_workspace_bytes(4096, 1000, torch.bfloat16, True),
                               dtype=torch.uint8, device=DEV)
    return o


def _step(wsf, t, o, s):
    eps = 2.0 ** -17
    wsf.ws_fwd(t["x"], t["w"], y=o["y"], stream=s)
    wsf.ws_bwd(t["x"], t["w"], t["dyv"], dx=o["dx"], grad_w=o["gw"], workspace=o["ws_ws"], stream=s)
    wsf.silu_fwd(t["xs"], t["ws"], y=o["ys"], stream=s)
    wsf.silu_bwd(t["dys"], t["xs"], t["ws"], dx=o["dxs"], dw=o["dws"], workspace=o["silu_ws"], stream=s)
    wsf.softmax_fwd(t["x"], y=o["ym"], stream=s)
    wsf.softmax_bwd(o["ym"], t["dyn"], dx=o["dxm"], stream=s)
    wsf.layernorm_fwd(t["x"], t["wn"], t["bn"], eps, y=o["yn"], stream=s)
    wsf.layernorm_bwd(t["x"], t["wn"], t["dyn"], eps, dx=o["dxn"], grad_w=o["gwn"], grad_b=o["gbn"],
                      workspace=o["norm_ws"], stream=s)


def test_capture_and_replay_match_eager(wsf):
    t = _tensors()
    eager = _outputs(wsf, t)
    s = torch.cuda.Stream(device=DEV)
    with torch.cuda.stream(s):
        _step(wsf, t, eager, s)
    s.synchronize()
    o = _outputs(wsf, t)
    for v in o.values():
        v.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step(wsf, t, o, s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for k in eager:
        if k.endswith("_ws"):
            continue
        assert torch.equal(o[k], eager[k]), k
    # new inputs in place: the replay follows them
    t["x"].mul_(0.5)
    t["dys"].neg_()
    with torch.cuda.stream(s):
        _step(wsf, t, eager, s)
    s.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for k in eager:
        if k.endswith("_ws"):
            continue
        assert torch.equal(o[k], eager[k]), k


def test_capture_cluster_paths(wsf):
    # wide rows take thread-block clusters (and fp32 rows of 140,000 the
    # two-pass cluster kernels); run alone, this test makes the
    # first use of the fp16 softmax cluster kernels inside the capture (their
    # one-time occupancy query and kernel attributes happen there), while the
    # bf16 norm kernels were used eagerly before
    g = torch.Generator(device=DEV).manual_seed(1)
    eps = 2.0 ** -17
    x16 = torch.randn(64, 36000, device=DEV, generator=g).half()
    dy16 = torch.randn(64, 36000, device=DEV, generator=g).half()
    x32 = torch.randn(6, 140000, device=DEV, generator=g)  # two-pass rows
    dy32 = torch.randn(6, 140000, device=DEV, generator=g)
    xb = torch.randn(300, 20000, device=DEV, generator=g).bfloat16()
    dyb = torch.randn(300, 20000, device=DEV, generator=g).bfloat16()
    wn = 1 + 0.1 * torch.randn(20000, device=DEV, generator=g)
    bn = 0.1 * torch.randn(20000, device=DEV, generator=g)
    wsf.rmsnorm_fwd(xb, wn, eps)
    wsf.layernorm_bwd(xb, wn, dyb, eps)
    torch.cuda.synchronize()

    def outs():
        return {"ym": torch.empty_like(x16), "dxm": torch.empty_like(x16),
                "y2": torch.empty_like(x32), "dx2": torch.empty_like(x32),
                "yn": torch.empty_like(xb), "dxn": torch.empty_like(xb),
                "gw": torch.empty(20000, device=DEV), "gb": torch.empty(20000, device=DEV),
                "ws": torch.empty(wsf.norm_bwd_workspace_bytes(300, 20000, torch.bfloat16, True),
                                  dtype=torch.uint8, device=DEV)}

    def step(o, s):
        wsf.softmax_fwd(x16, y=o["ym"], stream=s)
        wsf.softmax_bwd(o["ym"], dy16, dx=o["dxm"], stream=s)
        wsf.softmax_fwd(x32, y=o["y2"], stream=s)
        wsf.softmax_bwd(o["y2"], dy32, dx=o["dx2"], stream=s)
        wsf.layernorm_fwd(xb, wn, bn, eps, y=o["yn"], stream=s)
        wsf.layernorm_bwd(xb, wn, dyb, eps, dx=o["dxn"], grad_w=o["gw"], grad_b=o["gb"],
                          workspace=o["ws"], stream=s)

    s = torch.cuda.Stream(device=DEV)
    o = outs()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        step(o, s)
    gr.replay()
    torch.cuda.synchronize()
    eager = outs()
    with torch.cuda.stream(s):
        step(eager, s)
    s.synchronize()
    for k in eager:
        if k != "ws":
            assert torch.equal(o[k], eager[k]), k
    assert wsf.cluster_wait_timeouts() == 0
