"""Shared helpers of the GPU tests: build a seeded layer case on the device, run the library
through its C ABI, and compare with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

TOL_REL, TOL_ABS = 2e-2, 1e-3      # max|err| <= 2e-2 * max|ref| + 1e-3


def lib():
    from sparse_expert_ffn_layer_gb300 import _build
    _build.build()
    import sparse_expert_ffn_layer_gb300 as m
    return m


def within_tol(got: np.ndarray, ref: np.ndarray):
    err = float(np.max(np.abs(got.astype(np.float64) - ref))) if ref.size else 0.0
    bound = TOL_REL * (float(np.max(np.abs(ref))) if ref.size else 0.0) + TOL_ABS
    return err <= bound, err, bound


def torch_dtype(cfg):
    return torch.float32 if cfg.dtype == "f32" else torch.float16


class Case:
    """Seeded inputs of one layer call: host copies of what the oracle needs, device tensors."""

    def __init__(self, cfg, T, seed=0, batch=0, tokens=None, Wg=None):
        self.cfg, self.T, self.seed = cfg, T, seed
        dt = synth.F32 if cfg.dtype == "f32" else synth.F16
        self.tokens = tokens if tokens is not None else synth.fill(
            (T, cfg.d), dt, seed, synth.TID_TOKENS + (batch << 8), cfg.tok_sigma)
        if Wg is None:
            cs = synth.gate_col_scale(cfg, seed)
            Wg = synth.fill((cfg.d, cfg.E), synth.F32, seed, synth.TID_WG, cfg.w_sigma, col_scale=cs)
        self.Wg = Wg
        tdt = torch_dtype(cfg)
        self.d_tokens = torch.from_numpy(self.tokens).cuda()
        self.d_Wg = torch.from_numpy(self.Wg).cuda()
        self.d_W1 = torch.empty((cfg.E, cfg.d, cfg.f), dtype=tdt, device="cuda")
        self.d_W2 = torch.empty((cfg.E, cfg.f, cfg.d), dtype=tdt, device="cuda")
        synth.fill_cuda(self.d_W1, seed, synth.TID_W1, cfg.w_sigma)
        synth.fill_cuda(self.d_W2, seed, synth.TID_W2, cfg.w_sigma)
        self.Wr1 = self.Wr2 = self.d_Wr1 = self.d_Wr2 = None
        if cfg.residual:
            self.Wr1 = synth.fill((cfg.d, cfg.f_res), dt, seed, synth.TID_WR1, cfg.w_sigma)
            self.Wr2 = synth.fill((cfg.f_res, cfg.d), dt, seed, synth.TID_WR2, cfg.w_sigma)
            self.d_Wr1 = torch.from_numpy(self.Wr1).cuda()
            self.d_Wr2 = torch.from_numpy(self.Wr2).cuda()
        torch.cuda.synchronize()
        self._routing = None

    @property
    def mlp_type(self):
        return 1 if self.cfg.residual else 0

    def workspace(self, m):
        n = m.moe_workspace_size(self.T, self.cfg.d, self.cfg.f, self.cfg.E, self.cfg.k, self.cfg.cf,
                                 self.mlp_type, self.cfg.f_res, 0 if self.cfg.dtype == "f32" else 1)
        return torch.empty(n, dtype=torch.uint8, device="cuda")

    def forward(self, m, ws=None):
        cfg = self.cfg
        out = torch.full((self.T, cfg.d), float("nan"), dtype=torch_dtype(cfg), device="cuda")
        idx = torch.full((self.T, cfg.k), -7, dtype=torch.int32, device="cuda")
        slot = torch.full((self.T, cfg.k), -7, dtype=torch.int32, device="cuda")
        ws = self.workspace(m) if ws is None else ws
        m.moe_layer_forward(self.d_tokens, self.d_Wg, self.d_W1, self.d_W2, cfg.k, cfg.cf, out, ws,
                            mlp_type=self.mlp_type, Wr1=self.d_Wr1, Wr2=self.d_Wr2,
                            topk_idx_out=idx, slot_of_out=slot)
        st = m.moe_status_read(ws)
        assert st == m.MOE_OK, m.moe_status_string(st)
        return out.float().cpu().numpy(), idx.cpu().numpy(), slot.cpu().numpy()

    def routing(self):
        if self._routing is None:
            # the ABI takes cf as binary32: give the oracle that value
            self._routing = oracle.route(self.tokens, self.Wg, self.cfg.k,
                                         float(np.float32(self.cfg.cf)))
        return self._routing

    def reference_rows(self, rows, max_experts=24):
        """Oracle output of the listed rows.  Rows are taken in groups whose kept assignments
        use at most max_experts experts, so that only those experts' weights are drawn on the
        host at a time (the largest layers hold 26 GB of expert weights)."""
        r = self.routing()
        rows = np.asarray(rows, dtype=np.int32)
        need = [sorted({int(r.topk_idx[t, j]) for j in range(self.cfg.k)
                        if r.disp.slot_of[t, j] >= 0}) for t in rows]
        order = sorted(range(rows.size), key=lambda i: (need[i] or [-1])[0])
        out = np.empty((rows.size, self.cfg.d), np.float64)

        def flush(group, experts):
            if not group:
                return
            w1, w2 = synth.expert_slices(self.cfg, sorted(experts), self.seed)
            out[group] = oracle.combine_rows(self.tokens, r, w1, w2, self.Wr1, self.Wr2,
                                             rows=rows[group])

        group, experts = [], set()
        for i in order:
            union = experts | set(need[i])
            if len(union) > max_experts and group:
                flush(group, experts)
                group, union = [], set(need[i])
            group.append(i)
            experts = union
        flush(group, experts)
        return out


def sample_rows(r, T, n_random=512, seed=0, n_dropped=64):
    """Rows compared at sizes where the oracle cannot take every row: the first and last
    tokens, up to n_dropped tokens with a dropped assignment, for every active expert the
    first and the last token it kept (the last one sits at the capacity boundary), and
    n_random random tokens."""
    rng = np.random.default_rng(seed)
    rows = {0, T - 1}
    dropped = np.where((r.disp.slot_of < 0).any(axis=1))[0]
    rows.update(dropped[:n_dropped].tolist())
    offs, perm = r.disp.offsets, r.disp.perm
    for e in range(offs.size - 1):
        if offs[e + 1] > offs[e]:
            rows.add(int(perm[offs[e]]))
            rows.add(int(perm[offs[e + 1] - 1]))
    rows.update(rng.choice(T, size=min(T, n_random), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int32)
