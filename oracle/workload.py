"""Host-side builders of oracle inputs for the synthetic workloads: masters
from gen/, quantised by the oracle itself. TEST INFRASTRUCTURE ONLY."""
import numpy as np

from gen import gen
from . import oracle as orc


class OracleLayer:
    """One MoE layer as the oracle sees it; experts are quantised on demand."""

    def __init__(self, seed, layer, H, I, S, E, bias_range):
        self.seed, self.layer, self.H, self.I, self.S, self.E = seed, layer, H, I, S, E
        self.Wg = gen.router_w(seed, layer, E, H)
        self.bias = gen.router_bias(seed, layer, E, *bias_range)
        self.sh_up = orc.Mat.from_master(gen.sh_up_master(seed, layer, S, H))
        self.sh_down = orc.Mat.from_master(gen.sh_down_master(seed, layer, H, S))
        self.up, self.down = {}, {}

    def ensure(self, experts):
        for e in sorted(set(int(x) for x in np.asarray(experts).reshape(-1))):
            if e not in self.up:
                self.up[e] = orc.Mat.from_master(gen.up_master(self.seed, self.layer, e, self.I, self.H))
                self.down[e] = orc.Mat.from_master(gen.down_master(self.seed, self.layer, e, self.H, self.I))

    def route(self, h, k, rms_eps=0.0):
        x = orc.rms_norm(h, rms_eps) if rms_eps > 0 else h
        r = orc.route(x, self.Wg, self.bias, k)
        if rms_eps > 0:
            r["zslack"] = orc.rms_norm_slack(h, rms_eps, self.Wg)
        return r

    def forward(self, h, k, w4a4, residual, routing=None, rms_eps=0.0):
        """One MoE block: x = RMSNorm(h) when rms_eps > 0 (else x = h), route(x),
        experts(x), plus h when residual."""
        x = orc.rms_norm(h, rms_eps) if rms_eps > 0 else h
        if routing is None:
            r = orc.route(x, self.Wg, self.bias, k)
            if rms_eps > 0:
                r["zslack"] = orc.rms_norm_slack(h, rms_eps, self.Wg)
        else:
            r = routing
        self.ensure(r["idx"])
        out, outf = orc.moe_layer(x, r["idx"], r["w"], self.up, self.down, self.sh_up,
                                  self.sh_down, w4a4, h if residual else None, self.E)
        return out, outf, r


def lm_head_mat(seed, V, H):
    return orc.Mat.from_master(gen.lm_head_master(seed, V, H))
