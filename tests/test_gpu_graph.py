"""The step captured in a CUDA graph and replayed, against eager launches.

Every run-time input of a step is a device pointer (lr, step count, loss scale,
found-inf flag) and the plan never changes after creation, so the non-finite
check and the step can be captured once and replayed with new grads and a new
learning rate written into the same buffers.  "Support store_param_remainders
feature from Apex in TE Fused Adam #1408" reports that its capturable mode and
remainders could not be combined; here the bf16 + remainder mode is captured
too.  Replays must match eager steps bit for bit, skipped steps included.
"""

import numpy as np
import pytest
import torch

from adamw_optimizer_step_tensor_gb300 import FusedAdamW

pytestmark = pytest.mark.gpu
SIZES = [4099, 70000, 33]


def _state(mode, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = []
    for n in SIZES:
        d = {"m": torch.zeros(n, device="cuda"), "v": torch.zeros(n, device="cuda"),
             "g": torch.zeros(n, dtype=torch.float16, device="cuda")}
        if mode == "fp32":
            d["p"] = torch.randn(n, generator=g, device="cuda") * 0.02
            d["r"] = None
        else:
            d["p"] = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
            d["r"] = torch.randint(0, 1 << 15, (n,), generator=g, device="cuda").to(torch.int16)
        out.append(d)
    return out


def _opt(state, mode):
    return FusedAdamW([d["p"] for d in state], [d["g"] for d in state], [d["m"] for d in state],
                      [d["v"] for d in state], [0.1, 0.0, 0.1], mode=mode,
                      param_rems=[d["r"] for d in state] if mode == "bf16_rem" else None)


@pytest.mark.parametrize("mode", ["fp32", "bf16_rem"])
def test_graph_replay_matches_eager(mode):
    eager_state, graph_state = _state(mode, 3), _state(mode, 3)
    eager, graphed = _opt(eager_state, mode), _opt(graph_state, mode)
    scalars = {}
    for name in ("eager", "graph"):
        scalars[name] = dict(lr=torch.tensor([1e-3], device="cuda"),
                             step=torch.zeros(1, dtype=torch.int32, device="cuda"),
                             scale=torch.tensor([1024.0], device="cuda"),
                             found=torch.zeros(1, device="cuda"))

    def run(opt, sc):
        opt.check_nonfinite(sc["found"])
        opt.step(sc["lr"], sc["step"], grad_scale=sc["scale"], found_inf=sc["found"])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run(graphed, scalars["graph"])
    torch.cuda.synchronize()

    rng = np.random.default_rng(4)
    for it in range(12):
        lr = float(np.float32(1e-3 * (0.9 ** it)))
        for d_e, d_g in zip(eager_state, graph_state):
            x = torch.from_numpy((rng.normal(0, 1e-3, d_e["g"].numel()) * 1024).astype(np.float16))
            d_e["g"].copy_(x)
            d_g["g"].copy_(x)
        if it in (4, 9):
            eager_state[1]["g"][77] = float("nan")
            graph_state[1]["g"][77] = float("nan")
        scalars["eager"]["lr"].fill_(lr)
        scalars["graph"]["lr"].fill_(lr)
        run(eager, scalars["eager"])
        graph.replay()
        torch.cuda.synchronize()
        assert int(scalars["eager"]["step"].item()) == int(scalars["graph"]["step"].item())
        bad = []
        for i, (d_e, d_g) in enumerate(zip(eager_state, graph_state)):
            for k in ("p", "r", "m", "v"):
                if d_e[k] is not None:
                    a = d_e[k].view(torch.int16 if d_e[k].element_size() == 2 else torch.int32)
                    b = d_g[k].view(torch.int16 if d_g[k].element_size() == 2 else torch.int32)
                    diff = torch.nonzero(a != b).flatten().cpu().numpy()
                    if diff.size:
                        bad.append(f"tensor {i} {k}: {diff.size} of {a.numel()} differ, "
                                   f"[{diff[0]}, {diff[-1]}]")
        assert not bad, (it, int(scalars["eager"]["step"].item()), bad)
    assert int(scalars["graph"]["step"].item()) == 10


def test_graph_walks_a_device_lr_schedule():
    """lookup(table[step]) + step captured once; each replay takes the next cosine entry."""
    import synth
    from adamw_optimizer_step_tensor_gb300 import _capi as C
    from oracle import adamw as OA

    n = 20000
    rng = np.random.default_rng(9)
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    grads = [rng.normal(0, 1e-3, n).astype(np.float32) for _ in range(7)]
    table = torch.tensor([OA.f32(synth.cosine_lr(s, total=7)) for s in range(7)], device="cuda")
    p = torch.from_numpy(p0.copy()).cuda()
    g = torch.zeros(n, device="cuda")
    m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    opt = FusedAdamW([p], [g], [m], [v], [0.1])
    lr = torch.zeros(1, device="cuda")
    step = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        s = torch.cuda.current_stream().cuda_stream
        C.adamw_lr_from_table(table.data_ptr(), 7, step.data_ptr(), lr.data_ptr(), s)
        opt.step(lr, step)
    torch.cuda.synchronize()
    ref = OA.Tensor(p=p0.copy(), g=None, m=np.zeros(n, np.float32), v=np.zeros(n, np.float32),
                    wd=OA.f32(0.1))
    for t in range(1, 8):
        g.copy_(torch.from_numpy(grads[t - 1]))
        graph.replay()
        ref.g = grads[t - 1]
        OA.step_f32([ref], lr=OA.f32(synth.cosine_lr(t - 1, total=7)), beta1=OA.f32(0.9),
                    beta2=OA.f32(0.999), eps=OA.f32(1e-8), t=t)
        torch.cuda.synchronize()
        assert float(lr.item()) == OA.f32(synth.cosine_lr(t - 1, total=7))
        assert np.array_equal(p.cpu().numpy().view(np.uint32), ref.p.view(np.uint32)), t
    assert int(step.item()) == 7


def _build_kind(kind, seed):
    """Two identical optimizers of one kind (state on the device), and a step function."""
    sizes = [4099, 70_000, 33 * 64]
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    st = []
    for n in sizes:
        d = {"p": torch.randn(n, generator=g, device="cuda") * 0.02,
             "g": torch.zeros(n, dtype=torch.float16, device="cuda"),
             "m": torch.zeros(n, device="cuda")}
        if kind in ("q8", "q4"):
            nb = (n + (255 if kind == "q8" else 127)) // (256 if kind == "q8" else 128)
            nc = n if kind == "q8" else (n + 1) // 2
            d.update(m=torch.zeros(nc, dtype=torch.uint8, device="cuda"),
                     v=torch.zeros(nc, dtype=torch.uint8, device="cuda"),
                     am=torch.zeros(nb, device="cuda"), av=torch.zeros(nb, device="cuda"))
        elif kind == "mini":
            d["v"] = torch.zeros(n // (n if n != 33 * 64 else 64), device="cuda")
        elif kind in ("ademamix",):
            d["v"] = torch.zeros(n, device="cuda")
            d["m2"] = torch.zeros(n, device="cuda")
        elif kind not in ("lion", "rmsprop"):
            d["v"] = torch.zeros(n, device="cuda")
        st.append(d)
    kw = {}
    if kind in ("q8", "q4"):
        kw = dict(mode=kind, absmax_m=[d["am"] for d in st], absmax_v=[d["av"] for d in st])
    if kind == "ademamix":
        kw = dict(exp_avg_slows=[d["m2"] for d in st])
    if kind == "mini":
        kw = dict(v_blocks=[4099, 70_000, 64])
    opt = FusedAdamW([d["p"] for d in st], [d["g"] for d in st], [d["m"] for d in st],
                     [d.get("v") for d in st] if "v" in st[0] else None, [0.1, 0.0, 0.1], **kw)

    def step(sc):
        opt.check_nonfinite(sc["found"])
        args = dict(grad_scale=sc["scale"], found_inf=sc["found"])
        if kind == "lion":
            opt.step_lion(sc["lr"], sc["step"], **args)
        elif kind == "rmsprop":
            opt.step_coupled("rmsprop", sc["lr"], sc["step"], beta=0.99, **args)
        elif kind == "ademamix":
            opt.step_ademamix(sc["lr"], sc["step"], **args)
        elif kind == "mini":
            opt.step_mini(sc["lr"], sc["step"], **args)
        else:
            opt.step(sc["lr"], sc["step"], **args)
    return st, opt, step


@pytest.mark.parametrize("kind", ["lion", "rmsprop", "ademamix", "mini", "q8", "q4"])
def test_graph_replay_matches_eager_for_every_rule(kind):
    st_e, opt_e, step_e = _build_kind(kind, 5)
    st_g, opt_g, step_g = _build_kind(kind, 5)
    sc = {name: dict(lr=torch.tensor([1e-3], device="cuda"), step=torch.zeros(1, dtype=torch.int32, device="cuda"),
                     scale=torch.tensor([1024.0], device="cuda"), found=torch.zeros(1, device="cuda"))
          for name in ("e", "g")}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step_g(sc["g"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    for it in range(6):
        for a, b in zip(st_e, st_g):
            x = torch.from_numpy((rng.normal(0, 1e-3, a["g"].numel()) * 1024).astype(np.float16))
            a["g"].copy_(x)
            b["g"].copy_(x)
        if it == 3:
            st_e[1]["g"][5] = float("inf")
            st_g[1]["g"][5] = float("inf")
        for name in ("e", "g"):
            sc[name]["lr"].fill_(float(np.float32(1e-3 * 0.8 ** it)))
        step_e(sc["e"])
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(st_e, st_g):
            for k in a:
                if k == "g":
                    continue
                x, y = a[k], b[k]
                assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), (kind, it, k)
    assert int(sc["g"]["step"].item()) == int(sc["e"]["step"].item()) == 5
