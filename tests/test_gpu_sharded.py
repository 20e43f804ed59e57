"""Entry-sharded CSA decode on one GPU with virtual shards (slices of one cache), through the C
ABI: every shard's candidates (csa_shard_candidates), their merge (csa_topk_merge) and the LSE
merge of the shards' attention outputs (csa_lse_merge) against the unsharded selection (bit for
bit, and the fp64 oracle's) and the oracle's attention output (max-abs 1e-2, relative L2 5e-3).
Shards are even and uneven, and one case puts every selected entry in one shard (the others
contribute empty attention sets)."""
import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
from long_context_compressed_pooling_b300 import sharded
from synth import LayerShape, generate_layer
from _helpers import assert_attention_close, assert_lse_close, bits, f64, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_status():
    if torch.cuda.is_available():
        csa.device_status(reset=True)
    yield
    if torch.cuda.is_available():
        assert csa.device_status(reset=True) == 0


def _layer(B, N, m, k, W, seed, skew=False):
    s = LayerShape("csa", B=B, N=N, Nq=1, q_pos0=N - 1, H=64, d=128, m=m, W=W, k=k, H_I=4,
                   d_I=64, q_scale=1.0 / np.sqrt(128), compress_begin=0)
    x = generate_layer(s, seed=seed, device=DEV)
    E = N // m
    if skew:  # the largest scores all in the first eighth of the entries
        x["ki_scales"][:] = 123
        x["ki_scales"][:, : E // 8] = 127
    kc = torch.empty((B, E, 128), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc)
    return x, kc, vc


@pytest.mark.parametrize("B,N,k,W,cuts,skew", [
    (2, 65536, 512, 128, [0, 4096, 8192, 12288, 16384], False),   # 4 even shards
    (3, 40000, 300, 64, [0, 1000, 7000, 10000], False),           # 3 uneven shards
    (2, 65536, 256, 128, [0, 8192, 16384], True),                 # one shard holds the top-k
    (1, 8192, 64, 0, [0, 512, 1024, 1536, 2048], False),          # no window
])
def test_sharded_decode_matches_unsharded(B, N, k, W, cuts, skew):
    m = 4
    x, kc, vc = _layer(B, N, m, k, W, seed=N + k, skew=skew)
    t = N - 1
    shards = []
    for s in range(len(cuts) - 1):
        a, e = cuts[s], cuts[s + 1]
        last = s == len(cuts) - 2
        shards.append(sharded.Shard(
            base=a, qi_codes=x["qi_codes"], qi_scales=x["qi_scales"],
            ki_codes=x["ki_codes"][:, a:e].contiguous(), ki_scales=x["ki_scales"][:, a:e].contiguous(),
            k_cmp=kc[:, a:e].contiguous(), v_cmp=vc[:, a:e].contiguous(), q=x["q"],
            k_raw=x["k_raw"] if last else None, v_raw=x["v_raw"] if last else None))
    idx, cnt, out, lse = sharded.decode_step(shards, t, m, k, W)
    torch.cuda.synchronize()
    # the unsharded selection on the GPU: identical
    ridx, rcnt, _ = csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"],
                                   t, m, k)
    assert torch.equal(idx, ridx[:, 0]) and torch.equal(cnt, rcnt[:, 0])
    E = N // m
    for b in range(B):
        qb, kr, vr = bits(x["q"][b]), bits(x["k_raw"][b]), bits(x["v_raw"][b])
        ref = O.csa_layer_seq(qb, kr, vr, npy(x["logits"][b]), npy(x["qi_codes"][b]),
                              npy(x["qi_scales"][b]), npy(x["ki_codes"][b]),
                              npy(x["ki_scales"][b]), m=m, W=W, k=k, d_I=64, q_pos0=t,
                              k_cmp=f64(kc[b]), v_cmp=f64(vc[b]))
        np.testing.assert_array_equal(npy(idx[b]), ref["idx"][0])
        assert int(cnt[b]) == int(ref["cnt"][0])
        assert_attention_close(f64(out[b]), ref["out"][0], f"b={b}")
        assert_lse_close(npy(lse[b]), ref["lse"][0], f"b={b}")


def test_lse_merge_of_empty_and_single_parts():
    # two parts, the second empty (lse -inf): the merge is the first part; all empty gives 0
    S, R, d = 2, 5, 128
    g = torch.Generator(device=DEV).manual_seed(3)
    parts = torch.randn((S, R, d), generator=g, device=DEV).to(torch.bfloat16)
    lses = torch.randn((S, R), generator=g, device=DEV)
    lses[1] = -float("inf")
    lses[0, 4] = -float("inf")
    out, lse = csa.lse_merge(parts, lses, want_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out[:4], parts[0, :4])
    assert torch.all(out[4].float() == 0) and torch.isneginf(lse[4])
    assert torch.allclose(lse[:4], lses[0, :4])
