"""moe_route_topk on the GPU against the oracle: indices bit-exact (a swap
is accepted only between experts whose exact biased scores lie within their
binary32 error bounds), gate weights to 1e-5."""
import numpy as np
import pytest
import torch

from gen import gen
from oracle import oracle as orc
from tests.gpu_fixtures import nm  # noqa: F401
from tests.helpers import check_routing, to_dev_bf16

pytestmark = pytest.mark.gpu


def run(nm, h, Wg, bias, k):
    idx, w = nm.moe_route_topk(to_dev_bf16(h), torch.from_numpy(Wg).cuda(),
                               torch.from_numpy(bias).cuda(), k)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,k,H,brange", [
    (1, 128, 6, 2688, 0.1), (4, 128, 6, 2688, 0.1), (37, 128, 6, 2688, 0.1),
    (1024, 128, 6, 2688, 0.5), (256, 128, 6, 2688, 0.1), (3, 16, 4, 256, 0.1),
    (2, 8, 8, 64, 0.1), (5, 256, 32, 128, 0.1), (9, 33, 1, 96, 0.1)])
def test_route_matches_oracle(nm, T, E, k, H, brange):
    h = gen.hidden_bf16(T, H, 0, layer=0)
    Wg = gen.router_w(0, 0, E, H)
    bias = gen.router_bias(0, 0, E, -brange, brange)
    gi, gw = run(nm, h, Wg, bias, k)
    r = orc.route(h, Wg, bias, k)
    exempt = check_routing(gi, gw, r, k)
    assert exempt <= max(1, T // 100)


def test_zero_hidden_selects_by_bias(nm):
    E, H, k = 128, 2688, 6
    Wg = gen.router_w(0, 1, E, H)
    bias = gen.router_bias(0, 1, E, -0.1, 0.1)
    h = np.zeros((2, H), np.uint16)
    gi, gw = run(nm, h, Wg, bias, k)
    order = np.argsort(-bias.astype(np.float64), kind="stable")[:k]
    assert (gi == order[None, :]).all()
    assert np.allclose(gw, 1.0 / k, rtol=1e-6)
