"""A PR-MoE pyramid stack on the GPU: layers chained through device buffers and replayed as
one CUDA graph, against the oracle's chain of the same layers.

Between layers the two chains differ by rounding (each layer's output is rounded to fp16 on
both sides, from slightly different fp32 / float64 values), so a token whose top-1 margin at
some layer is below the logits' error bound may legitimately pick the other expert.  Such a
flip is accepted only when the oracle's margin is within the bound that the input difference
implies, and the token is not compared after it; every other token must match at every layer.
The layers are dropless, so a flip cannot change another token's capacity decision.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from moe_cases import lib, within_tol

pytestmark = pytest.mark.gpu


def _host_layer(cfg, seed):
    cs = synth.gate_col_scale(cfg, seed)
    return dict(
        Wg=synth.fill((cfg.d, cfg.E), synth.F32, seed, synth.TID_WG, cfg.w_sigma, col_scale=cs),
        W1=synth.fill((cfg.E, cfg.d, cfg.f), synth.F16, seed, synth.TID_W1, cfg.w_sigma),
        W2=synth.fill((cfg.E, cfg.f, cfg.d), synth.F16, seed, synth.TID_W2, cfg.w_sigma),
        Wr1=synth.fill((cfg.d, cfg.f_res), synth.F16, seed, synth.TID_WR1, cfg.w_sigma),
        Wr2=synth.fill((cfg.f_res, cfg.d), synth.F16, seed, synth.TID_WR2, cfg.w_sigma))


@pytest.mark.parametrize("T", [64, 37, 300])
def test_pyramid_stack_in_one_graph_matches_oracle_chain(T):
    m = lib()
    cfgs = [synth.CONFIGS[n] for n in synth.STACKS["tiny_pyramid_3"]]
    seed = 5
    d = cfgs[0].d
    host = [_host_layer(c, synth.layer_seed(seed, l)) for l, c in enumerate(cfgs)]
    dev = [{k: torch.from_numpy(v).cuda() for k, v in L.items()} for L in host]
    x0 = synth.fill((T, d), synth.F16, seed, synth.TID_TOKENS, 1.0)
    bufs = [torch.from_numpy(x0).cuda()] + [torch.empty((T, d), dtype=torch.float16, device="cuda")
                                            for _ in cfgs]
    idx = [torch.empty((T, c.k), dtype=torch.int32, device="cuda") for c in cfgs]
    slot = [torch.empty((T, c.k), dtype=torch.int32, device="cuda") for c in cfgs]
    ws = torch.empty(max(m.moe_workspace_size(T, c.d, c.f, c.E, c.k, c.cf, m.MOE_MLP_RESIDUAL,
                                              c.f_res, m.MOE_F16) for c in cfgs),
                     dtype=torch.uint8, device="cuda")

    def run():
        for l, c in enumerate(cfgs):
            L = dev[l]
            m.moe_layer_forward(bufs[l], L["Wg"], L["W1"], L["W2"], c.k, c.cf, bufs[l + 1], ws,
                                mlp_type=m.MOE_MLP_RESIDUAL, Wr1=L["Wr1"], Wr2=L["Wr2"],
                                topk_idx_out=idx[l], slot_of_out=slot[l])

    run()                                     # first calls outside the capture
    torch.cuda.synchronize()
    for b in bufs[1:]:
        b.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        run()
    g.replay()
    torch.cuda.synchronize()
    assert m.moe_status_read(ws) == m.MOE_OK
    first = [b.clone() for b in bufs[1:]]
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(first, bufs[1:])), "replays differ"

    outs, ins, routings = oracle.stack_forward(x0, host, 1, float("inf"))
    gpu_in = [b.float().cpu().numpy().astype(np.float64) for b in bufs[:-1]]
    gpu_out = [b.float().cpu().numpy().astype(np.float64) for b in bufs[1:]]
    alive = np.ones(T, bool)
    for l, c in enumerate(cfgs):
        r = routings[l]
        gi = idx[l].cpu().numpy()
        assert np.all(slot[l].cpu().numpy() >= 0)                   # dropless
        Wg_abs = np.abs(host[l]["Wg"].astype(np.float64))
        for t in np.where(alive & (gi[:, 0] != r.topk_idx[:, 0]))[0]:
            top = np.sort(r.logits[t].astype(np.float64))[::-1]
            margin = top[0] - top[1]
            dx = np.abs(gpu_in[l][t] - ins[l][t].astype(np.float64))
            xin = np.abs(ins[l][t].astype(np.float64))
            bound = 2 * np.max(dx @ Wg_abs) + 4 * c.d * 2.0 ** -24 * np.max(xin @ Wg_abs)
            assert margin <= bound, f"layer {l} token {t}: margin {margin:.3e} > bound {bound:.3e}"
            alive[t] = False
        assert np.isfinite(gpu_out[l]).all()
        ok, err, bnd = within_tol(gpu_out[l][alive], outs[l][alive])
        assert ok, f"layer {l}: max err {err:.3e} > {bnd:.3e}"
    assert alive.sum() >= T - T // 8, f"{T - alive.sum()} routing flips"
    assert 0.1 < np.abs(gpu_out[-1]).mean() < 10.0                  # activations stay O(1)
