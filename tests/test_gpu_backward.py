"""GPU layer backward (moe_layer_backward) against the oracle's fp64 gradients
(which are pinned by central finite differences on the CPU), and a second,
tighter comparison against a model of the CUDA path's bf16 storage points
(``tests/gpu_rounding_model.py``, itself checked only against the oracle):

* exact oracle, per element |gpu - ref| <= 2e-2 |ref| + 8e-2 rms(ref): the
  GPU stores the pre-activations, h, the expert outputs, g dy, dA / dG and
  each expert's input-gradient rows in bf16 (each rounding at most 2^-9
  relative), and a weight-gradient element that is a sum of a few tokens'
  terms inherits one token's rounding error in full: replaying those
  roundings in fp64 on the CPU for the 96-token case gives a largest error of
  4.9 % of the gradient's RMS, on elements much smaller than the RMS;
* the storage-point model, per element
  |gpu - ref| <= 1e-2 |ref| + 3e-2 rms(ref): what is left is fp32
  accumulation order and the odd value that rounds the other way -- one
  bf16 ulp (2^-8 of it) of a per-expert input-gradient row that the sum
  over the K experts then cancels down (a row element near 2 contributes
  0.008 to a dx element near 0.01 in the 96-token case).
A missing term does not fit inside either bound: the router's share of dx
alone is ~36 % of dx's RMS here."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_rounding_model import backward_at_gpu_storage_points
from tests.gpu_util import Guarded, dev_bf16, guarded_workspace, host_bits, lib
from tests.inputs_filtered import filter_x

pytestmark = pytest.mark.gpu

EXACT = (2e-2, 8e-2)     # (rtol, atol as a fraction of the tensor's RMS)
MATCHED = (1e-2, 3e-2)


def close(name, got, ref, tol):
    RTOL, ATOL_RMS = tol
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    scale = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    bound = RTOL * np.abs(ref) + ATOL_RMS * scale
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d/%d out of tolerance (max err %.3g, rms %.3g); first %s: gpu %s ref %s"
                             % (name, int(bad.sum()), bad.size, float(np.nanmax(err)), scale,
                                idx.tolist(), [float(got[tuple(i)]) for i in idx],
                                [float(ref[tuple(i)]) for i in idx]))


def run_backward(cfg, L, dy, poison_ws=False):
    """moe_layer_backward with NaN-filled outputs, each the head of a larger
    buffer whose sentinel tail must survive (as must the workspace's)."""
    moe = lib()
    n, d, h = cfg.n_experts, cfg.dim, cfg.hidden
    nan = float("nan")
    g = dict(dx=Guarded((max(cfg.T, 1), d), torch.bfloat16, nan),
             dwg=Guarded((d, n), torch.float32, nan),
             dw1=Guarded((n, h, d), torch.float32, nan),
             dw3=Guarded((n, h, d), torch.float32, nan),
             dw2=Guarded((n, d, h), torch.float32, nan))
    ws, wsg = guarded_workspace(moe, cfg, backward=True)
    if poison_ws:
        # every byte past the control region 0xFF: bf16 NaN in every grouped
        # buffer, so a padding row that is read without being zeroed poisons
        # the weight gradients
        ws[65536:].fill_(0xFF)
    if cfg.T > 0:
        x, dyd = dev_bf16(L.x), dev_bf16(dy)
    else:
        x = dyd = torch.zeros((1, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_backward(cfg, x, dev_bf16(L.wg), dev_bf16(L.w1), dev_bf16(L.w3),
                           dev_bf16(L.w2), dyd, g["dx"].view, g["dwg"].view, g["dw1"].view,
                           g["dw3"].view, g["dw2"].view, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    for k, b in g.items():
        b.check(k)
    wsg.check("backward workspace")
    return dict(dx=orc.widen_bf16(host_bits(g["dx"].view[:cfg.T])),
                **{k: g[k].view.cpu().numpy() for k in ("dwg", "dw1", "dw3", "dw2")})


def check_backward(cfg, poison_ws=False):
    L = mi.make_layer(cfg)
    filter_x(cfg, L.x, L.wg, L.shift)
    dy = mi.gen_x(cfg.replace(seed=cfg.seed + 1))
    got = run_backward(cfg, L, dy, poison_ws)
    ref = orc.moe_layer_backward(L.x, L.wg, L.w1, L.w3, L.w2, cfg.top_k, dy)
    model = backward_at_gpu_storage_points(L.x, L.wg, L.w1, L.w3, L.w2, cfg.top_k, dy)
    for name in ("dx", "dwg", "dw1", "dw3", "dw2"):
        close(name, got[name], ref[name], EXACT)
        close(name + " (storage-point model)", got[name], model[name], MATCHED)


@pytest.mark.parametrize("T,n,K", [(96, 8, 2), (200, 8, 1), (150, 16, 2), (64, 40, 4), (7, 8, 2)])
def test_backward_matches_oracle(T, n, K):
    cfg = mi.Config("bwd", T=T, dim=256, hidden=256, n_experts=n, top_k=K, seed=46200 + T + n)
    check_backward(cfg)


def test_backward_wider_dims_and_ragged_groups():
    # dim 512, hidden 768: several 256-wide tiles per expert in every GEMM
    cfg = mi.Config("bwd", T=333, dim=512, hidden=768, seed=46300)
    check_backward(cfg)


def test_backward_top8_of_40_odd_tile_count():
    # fine-grained shape: top 8 of 40 experts (wide router), hidden 1792 = 7
    # tiles of 256, so every weight-side loop ends on an odd tile
    cfg = mi.Config("bwd", T=48, dim=512, hidden=1792, n_experts=40, top_k=8, seed=46306)
    check_backward(cfg)


def test_backward_groups_without_padding():
    # top 2 of 2 experts: both groups hold exactly T = 128 rows (two whole
    # 64-row blocks), so no padding row lies between them
    cfg = mi.Config("bwd", T=128, dim=256, hidden=256, n_experts=2, top_k=2, seed=46304)
    check_backward(cfg)


def test_backward_ignores_stale_workspace():
    # ragged groups (96 tokens, top 2 of 8) in a workspace full of NaN bytes
    cfg = mi.Config("bwd", T=96, dim=256, hidden=256, seed=46305)
    check_backward(cfg, poison_ws=True)


def test_backward_zero_tokens_gives_zero_weight_gradients():
    cfg = mi.Config("bwd", T=0, dim=256, hidden=256, seed=46301)
    L = mi.make_layer(cfg)
    got = run_backward(cfg, L, np.zeros((0, cfg.dim), np.uint16))
    for name in ("dwg", "dw1", "dw3", "dw2"):
        assert np.all(got[name] == 0), name


def test_backward_is_deterministic():
    cfg = mi.Config("bwd", T=120, dim=256, hidden=256, seed=46302)
    L = mi.make_layer(cfg)
    dy = mi.gen_x(cfg.replace(seed=46303))
    a = run_backward(cfg, L, dy)
    b = run_backward(cfg, L, dy)
    for name in a:
        assert np.array_equal(a[name], b[name]), name


def test_backward_full_dims_every_token():
    # T=1024 at Mixtral dims (dim 4096, hidden 14336, top 2 of 8): ~256 grouped
    # rows per expert.  Checked in full: dx of every token and dW_g (a sum over
    # every token's router gradient); sampled: the dW1 / dW3 rows and dW2
    # columns of 4 hidden units of every expert.
    cfg = mi.CONFIGS["prefill"].replace(name="bwd-1k", T=1024, seed=46320)
    L = mi.make_layer(cfg)
    filter_x(cfg, L.x, L.wg, L.shift)
    dy = mi.gen_x(cfg.replace(seed=cfg.seed + 1))
    got = run_backward(cfg, L, dy)
    ref = orc.moe_layer_backward(L.x, L.wg, L.w1, L.w3, L.w2, cfg.top_k, dy, weight_grads=False)
    close("dx", got["dx"], ref["dx"], EXACT)
    close("dwg", got["dwg"], ref["dwg"], EXACT)
    rng = np.random.default_rng(cfg.seed)
    for e in range(cfg.n_experts):
        units = np.sort(rng.choice(cfg.hidden, 4, replace=False))
        r = orc.expert_weight_grad_units(L.x, L.wg, L.w1, L.w3, L.w2, cfg.top_k, dy, e, units)
        close("dw1[%d] rows" % e, got["dw1"][e][units], r["dw1"], EXACT)
        close("dw3[%d] rows" % e, got["dw3"][e][units], r["dw3"], EXACT)
        close("dw2[%d] columns" % e, got["dw2"][e][:, units], r["dw2"], EXACT)


def test_backward_full_dims_sampled():
    # T=16384 at Mixtral dims (dim 4096, hidden 14336, top 2 of 8): ~4096 grouped
    # rows per expert, so every GEMM runs many token tiles per expert and the dX
    # GEMM walks each expert's rows in L2-sized blocks.  Checked: dx of 32
    # sampled tokens, and the dW1 / dW3 rows and dW2 columns of 4 sampled hidden
    # units of every expert (each a sum over all of that expert's tokens).
    # dW_g is a sum over all 16384 tokens' expert outputs, beyond what the fp64
    # oracle evaluates here; it is checked in full at T=1024 above.
    moe = lib()
    cfg = mi.CONFIGS["prefill"].replace(name="bwd-full", T=16384, seed=46310)
    L = mi.make_layer(cfg)
    filter_x(cfg, L.x, L.wg, L.shift)
    dy = mi.gen_x(cfg.replace(seed=cfg.seed + 1))
    n, d, h = cfg.n_experts, cfg.dim, cfg.hidden
    f32 = dict(dtype=torch.float32, device="cuda")
    dx = torch.full((cfg.T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dwg = torch.full((d, n), float("nan"), **f32)
    dw1 = torch.full((n, h, d), float("nan"), **f32)
    dw3 = torch.full((n, h, d), float("nan"), **f32)
    dw2 = torch.full((n, d, h), float("nan"), **f32)
    ws = moe.new_backward_workspace(cfg)
    moe.moe_layer_backward(cfg, dev_bf16(L.x), dev_bf16(L.wg), dev_bf16(L.w1), dev_bf16(L.w3),
                           dev_bf16(L.w2), dev_bf16(dy), dx, dwg, dw1, dw3, dw2, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    assert torch.isfinite(dwg).all()
    rng = np.random.default_rng(cfg.seed)
    rows = np.sort(rng.choice(cfg.T, 32, replace=False))
    ref = orc.moe_layer_backward(L.x[rows], L.wg, L.w1, L.w3, L.w2, cfg.top_k, dy[rows],
                                 weight_grads=False)
    got_dx = orc.widen_bf16(host_bits(dx[torch.as_tensor(rows, device="cuda")]))
    close("dx (sampled tokens)", got_dx, ref["dx"], EXACT)
    for e in range(n):
        units = np.sort(rng.choice(h, 4, replace=False))
        r = orc.expert_weight_grad_units(L.x, L.wg, L.w1, L.w3, L.w2, cfg.top_k, dy, e, units)
        u = torch.as_tensor(units, device="cuda")
        close("dw1[%d] rows" % e, dw1[e][u].cpu().numpy(), r["dw1"], EXACT)
        close("dw3[%d] rows" % e, dw3[e][u].cpu().numpy(), r["dw3"], EXACT)
        close("dw2[%d] columns" % e, dw2[e][:, u].cpu().numpy(), r["dw2"], EXACT)
