"""The grouped expert path (more than 4 tokens: prefill and high-concurrency
decode) against the oracle: moe_permute bit-exact against a stable sort of
the pairs by expert, and moe_expert_forward elementwise within
|err| <= 1e-2 + 2e-2 |ref|, at small shapes over every token and at the
pages' layer shape (1024-token prefill with skewed expert loads, 256
concurrent tokens) on sampled tokens, tokens being independent."""
import numpy as np
import pytest
import torch

from gen import configs, gen
from oracle.workload import OracleLayer
from tests.gpu_fixtures import dev_routing, device_layer, nm  # noqa: F401
from tests.helpers import assert_close, bf16_bits, bf16_to_f64, check_routing, to_dev_bf16

pytestmark = pytest.mark.gpu

SMALL = dict(E=16, H=256, I=128, S=192)


def permute_ref(idx, E):
    """Stable grouping of the flattened pairs by expert (the plain definition)."""
    flat = idx.reshape(-1).astype(np.int64)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    tiles = np.concatenate([[0], np.cumsum((counts + 63) // 64)]).astype(np.int32)
    return offsets, perm, inv, tiles


@pytest.mark.parametrize("T,k,E", [(1, 1, 8), (5, 4, 16), (100, 6, 128), (1024, 6, 128), (3000, 8, 256)])
def test_permute_exact(nm, T, k, E):
    rng = np.random.default_rng(T * 7 + k)
    # distinct experts per token, skewed towards low ids
    p = np.exp(-np.arange(E) / (E / 4.0))
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    offsets, perm, inv, tiles = nm.moe_permute(torch.from_numpy(idx).cuda(), E, with_tiles=True)
    torch.cuda.synchronize()
    ro, rp, ri, rt = permute_ref(idx, E)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)
    assert np.array_equal(tiles.cpu().numpy(), rt)
    assert nm.nvfp4_last_device_error() == 0


def run_grouped(nm, L, OL, h, k, w4a4, residual, rms_eps, sample=None, gpu_routing=False):
    """moe_expert_forward on all T tokens; compared with the oracle on `sample`
    (all tokens when None). Returns the number of tokens left out as near-ties."""
    T = h.shape[0]
    hd = to_dev_bf16(h)
    mode = nm.W4A4 if w4a4 else nm.W4A16
    rows = np.arange(T) if sample is None else np.asarray(sample)
    if gpu_routing:
        idx, w = nm.moe_route_topk(hd, L.router_w, L.router_b, k, rms_eps=rms_eps)
        torch.cuda.synchronize()
    else:
        idx, w = dev_routing(OL.route(h, k, rms_eps))
    ws = nm.make_workspace(L, T, k, mode)
    out = nm.moe_expert_forward(L, hd, idx, w, mode, residual=hd if residual else None, workspace=ws,
                                rms_eps=rms_eps)
    torch.cuda.synchronize()
    assert nm.nvfp4_last_device_error() == 0
    got = bf16_to_f64(bf16_bits(out))
    r = OL.route(h[rows], k, rms_eps)
    gi, gw = idx.cpu().numpy()[rows], w.cpu().numpy()[rows]
    keep = np.array([np.array_equal(gi[i], r["idx"][i]) for i in range(len(rows))])
    if gpu_routing:
        check_routing(gi, gw, r, k)  # every difference must be a near-tie
    sub = {key: (v[keep] if isinstance(v, np.ndarray) and v.shape[:1] == (len(rows),) else v)
           for key, v in r.items()}
    ref, _, _ = OL.forward(h[rows][keep], k, w4a4, residual, routing=sub, rms_eps=rms_eps)
    assert_close(got[rows][keep], bf16_to_f64(ref), "grouped layer output")
    # same workspace again: the same bits
    out2 = nm.moe_expert_forward(L, hd, idx, w, mode, residual=hd if residual else None, workspace=ws,
                                 rms_eps=rms_eps)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    return int((~keep).sum())


@pytest.fixture(scope="module")
def small_layer(nm):
    c = SMALL
    return (device_layer(nm, 3, 1, c["E"], c["H"], c["I"], c["S"], (-0.3, 0.3)),
            OracleLayer(3, 1, c["H"], c["I"], c["S"], c["E"], (-0.3, 0.3)))


@pytest.mark.parametrize("T", [5, 8, 33, 100])
@pytest.mark.parametrize("w4a4", [False, True])
@pytest.mark.parametrize("residual,eps", [(False, 0.0), (True, 1e-5)])
def test_small_grouped(nm, small_layer, T, w4a4, residual, eps):
    L, OL = small_layer
    h = gen.hidden_bf16(T, SMALL["H"], 3, layer=5)
    run_grouped(nm, L, OL, h, 4, w4a4, residual, eps)


@pytest.fixture(scope="module")
def full_layer_skewed(nm):
    c = configs.shape(3)
    L = device_layer(nm, c["seed"], 0, c["E"], c["H"], c["I"], c["S"], c["bias"])
    OL = OracleLayer(c["seed"], 0, c["H"], c["I"], c["S"], c["E"], c["bias"])
    return c, L, OL


def test_prefill_1024_tokens(nm, full_layer_skewed):
    """The 1024-token prefill layer (W4A4, bias U(-0.5, 0.5): skewed expert
    loads) with the GPU's own routing; 16 sampled tokens against the oracle."""
    c, L, OL = full_layer_skewed
    h = gen.hidden_bf16(c["T"], c["H"], c["seed"], layer=configs.HIDDEN_LAYER)
    sample = np.unique(np.concatenate([[0, 1, c["T"] - 1], np.random.default_rng(5).integers(0, c["T"], 13)]))
    left_out = run_grouped(nm, L, OL, h, c["K"], True, False, 0.0, sample=sample, gpu_routing=True)
    assert left_out <= 1


def test_256_tokens_prenorm(nm, full_layer_skewed):
    """256 concurrent tokens through one W4A4 layer with the pre-norm and the
    residual, as the 256-token configuration chains them; sampled tokens."""
    c, L, OL = full_layer_skewed
    h = gen.hidden_bf16(256, c["H"], c["seed"], layer=7)
    sample = np.random.default_rng(6).choice(256, 12, replace=False)
    left_out = run_grouped(nm, L, OL, h, c["K"], True, True, 1e-5, sample=sample, gpu_routing=True)
    assert left_out <= 1


def test_grouped_workspace_too_small(nm, small_layer):
    L, _ = small_layer
    T, k = 9, 4
    hd = to_dev_bf16(gen.hidden_bf16(T, SMALL["H"], 3, layer=5))
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda") + torch.arange(k, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), 0.25, dtype=torch.float32, device="cuda")
    need = nm.moe_expert_forward_workspace_size(L, T, k, nm.W4A4)
    ws = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(nm.NVFP4Error) as ei:
        nm.moe_expert_forward(L, hd, idx, w, nm.W4A4, workspace=ws)
    assert ei.value.status == 4


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("w4a4", [False, True])
def test_grouped_path_at_decode_sizes(nm, T, w4a4):
    """With nvfp4_set_decode_max_tokens(0) even 1..4 tokens take the grouped
    path (the backend choice the concurrency sweep measures); it matches the
    oracle like the decode kernels do."""
    from tests.test_gpu_moe import SMALL, run_layer
    from tests.gpu_fixtures import device_layer
    from oracle.workload import OracleLayer
    c = SMALL
    L = device_layer(nm, 7, 2, c["E"], c["H"], c["I"], c["S"], (-0.1, 0.1))
    OL = OracleLayer(7, 2, c["H"], c["I"], c["S"], c["E"], (-0.1, 0.1))
    h = gen.hidden_bf16(T, c["H"], 7, layer=2, rho=0.5)
    try:
        nm.nvfp4_set_decode_max_tokens(0)
        run_layer(nm, L, OL, h, 4, w4a4, True)
    finally:
        nm.nvfp4_set_decode_max_tokens(4)
