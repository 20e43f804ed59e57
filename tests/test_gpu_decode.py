"""Parity of the one-launch CSA decode step (indexer, top-k and sparse attention of one query
token per sequence in one kernel, one thread-block cluster per sequence) with the fp64 oracle.

The step runs through csa_hca_layer_pair with a CSA layer only (its decode path with 64 heads of
dim 128 or fewer) and through csa_index_topk (the same kernel without the attention). Shapes
cover: several entry tiles per CTA with a ragged tail, every visible entry selected (k at or
above the visible count), a single entry, no window, fewer heads than 64, scores whose
k-th largest lies far below the maximum (the exact radix select instead of the near-max
histogram), selections that all fall in one CTA's share of the entries (the attention runs then
read another CTA's list), and a block size of 1. Top-k lists are compared bit for bit,
attention outputs within max-abs 1e-2 and relative L2 5e-3, LSE within 2e-3."""
import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
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


def _layer(B, N, m, k, W, H, seed, skew=None):
    s = LayerShape("csa", B=B, N=N, Nq=1, q_pos0=N - 1, H=H, d=128, m=m, W=W, k=k, H_I=4,
                   d_I=64, q_scale=1.0 / np.sqrt(128), compress_begin=max(0, (N // m - 1) * m))
    x = generate_layer(s, seed=seed, device=DEV)
    E = N // m
    if skew == "far" and E > 0:
        # a few entries score 16x above the rest: fewer than k keys lie within 255 BF16 steps
        # of the maximum, so the threshold comes from the exact radix select
        x["ki_scales"][:] = 123
        x["ki_scales"][:, : min(E, 10)] = 127
    elif skew == "last" and E > 0:
        # the largest scores all sit in the last eighth of the entries
        x["ki_scales"][:] = 123
        x["ki_scales"][:, E - E // 8:] = 127
    kc = torch.empty((B, E, 128), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    if s.compress_begin > 0:
        csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, kc, vc, 0, s.compress_begin)
    layer = dict(x, m=m, W=W, k=k, q_pos0=N - 1, compress_begin=s.compress_begin, k_cmp=kc,
                 v_cmp=vc, out=torch.empty_like(x["q"]),
                 lse=torch.empty((B, 1, H), dtype=torch.float32, device=DEV),
                 topk_idx=torch.full((B, 1, k), -7, dtype=torch.int32, device=DEV),
                 topk_cnt=torch.full((B, 1), -7, dtype=torch.int32, device=DEV),
                 scores=torch.zeros((B, 1, E), dtype=torch.bfloat16, device=DEV))
    return s, x, layer


CASES = [
    # B, N, m, k, W, H, skew
    (3, 4096, 4, 64, 128, 64, None),      # 8 tiles: one or two per CTA
    (2, 40032, 4, 300, 128, 64, None),    # ragged last tile, runs of ~27 keys per CTA
    (16, 32768, 4, 512, 128, 64, None),   # the benchmark's batch and k at 1/4 of the context
    (2, 1024, 4, 512, 128, 64, None),     # every visible entry selected
    (2, 7, 4, 16, 128, 64, None),         # one entry: the window dominates
    (2, 8192, 4, 128, 0, 64, None),       # no window
    (2, 8192, 4, 100, 64, 16, None),      # 16 heads
    (2, 16384, 4, 64, 128, 64, "far"),    # exact radix select
    (2, 65536, 4, 2048, 128, 64, "last"), # every selected entry in one CTA's share
    (1, 2000, 1, 77, 32, 64, None),       # block size 1
]


@pytest.mark.parametrize("B,N,m,k,W,H,skew", CASES)
def test_decode_step_matches_oracle(B, N, m, k, W, H, skew):
    s, x, layer = _layer(B, N, m, k, W, H, seed=N + k + B, skew=skew)
    csa.layer_pair(layer, None)
    torch.cuda.synchronize()
    assert csa.device_status(reset=True) == 0
    E = N // m
    nv = O.visible_entries(N - 1, m, E)
    for b in range(B):
        qb, kr, vr = bits(x["q"][b]), bits(x["k_raw"][b]), bits(x["v_raw"][b])
        w = npy(x["logits"][b])
        ref = O.csa_layer_seq(qb, kr, vr, w, npy(x["qi_codes"][b]), npy(x["qi_scales"][b]),
                              npy(x["ki_codes"][b]), npy(x["ki_scales"][b]), m=m, W=W, k=k,
                              d_I=64, q_pos0=N - 1)
        assert int(npy(layer["topk_cnt"][b])[0]) == int(ref["cnt"][0]), b
        np.testing.assert_array_equal(npy(layer["topk_idx"][b, 0]), ref["idx"][0],
                                      err_msg=f"top-k b={b}")
        if nv > k:  # the scores are computed (not needed when everything is selected)
            np.testing.assert_array_equal(bits(layer["scores"][b, 0])[:nv], ref["scores"][0],
                                          err_msg=f"scores b={b}")
        # attention on the layer's own bf16 entries, and the whole layer on the oracle's pooling
        o, l = O.csa_attend_one(O.bf16_to_f64(qb[0]), f64(layer["k_cmp"][b]),
                                f64(layer["v_cmp"][b]), ref["idx"][0], int(ref["cnt"][0]),
                                O.bf16_to_f64(kr), O.bf16_to_f64(vr), N - 1, W)
        assert_attention_close(f64(layer["out"][b, 0]), o, f"out b={b}")
        assert_lse_close(npy(layer["lse"][b, 0]), l, f"lse b={b}")
        assert_attention_close(f64(layer["out"][b, 0]), ref["out"][0], f"layer b={b}")


@pytest.mark.parametrize("B,N,k,skew", [(4, 1048576, 2048, None), (5, 160000, 300, "far")])
def test_decode_index_topk_matches_oracle(B, N, k, skew):
    """csa_index_topk with one query per sequence: the one-launch kernel without the attention
    where each CTA's share of a row fits it (160000 tokens), the separate indexer and top-k
    kernels beyond (1M tokens, 4 rows); both bit-exact."""
    m = 4
    E = N // m
    s = LayerShape("csa", B=B, N=N, Nq=1, q_pos0=N - 1, H=64, d=128, m=m, W=128, k=k, H_I=4,
                   d_I=64, q_scale=1.0 / np.sqrt(128), compress_begin=N - m)
    x = generate_layer(s, seed=3 * N + k, device=DEV, skip=("q", "k_raw", "v_raw", "logits"))
    if skew == "far":
        x["ki_scales"][:] = 123
        x["ki_scales"][:, :10] = 127
    idx, cnt, sc = csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"],
                                  N - 1, m, k, want_scores=True)
    torch.cuda.synchronize()
    qc, qs, kc, ks = (npy(x[n]) for n in ("qi_codes", "qi_scales", "ki_codes", "ki_scales"))
    scb = bits(sc)
    for b in range(B):
        ref = O.f64_to_bf16_rne(O.index_scores(qc[b, 0], qs[b, 0], kc[b], ks[b], 64))
        np.testing.assert_array_equal(scb[b, 0], ref, err_msg=f"scores b={b}")
        ridx, rcnt = O.topk_select(ref, E, k)
        assert int(npy(cnt)[b, 0]) == rcnt
        np.testing.assert_array_equal(npy(idx)[b, 0], ridx, err_msg=f"top-k b={b}")


@pytest.mark.parametrize("B,N,H,k", [(3, 8192, 128, 100),     # 128 heads: selection without attention
                                     (2, 1048576, 64, 512)])  # 1M: scores over the whole GPU
def test_decode_layer_pools_in_the_selection_launch(B, N, H, k):
    """A decode layer the one-launch step does not take (more than 64 heads; entry shares above
    8192 per CTA) pools the block the token closes inside its scoring launch: the entry written
    there is bit-identical to csa_compress's, and the layer matches the oracle."""
    m, W = 4, 128
    s, x, layer = _layer(B, N, m, k, W, H, seed=N + H)
    E = N // m
    ref_k = torch.empty((B, E, 128), dtype=torch.bfloat16, device=DEV)
    ref_v = torch.empty_like(ref_k)
    csa.compress(x["k_raw"], x["v_raw"], x["logits"], m, ref_k, ref_v, E * m - m, E * m)
    layer["k_cmp"][:, E - 1] = 7.0  # poisoned: the step must write it
    layer["v_cmp"][:, E - 1] = 7.0
    csa.layer_pair(layer, None)
    torch.cuda.synchronize()
    assert csa.device_status(reset=True) == 0
    assert torch.equal(layer["k_cmp"][:, E - 1], ref_k[:, E - 1])
    assert torch.equal(layer["v_cmp"][:, E - 1], ref_v[:, E - 1])
    nv = O.visible_entries(N - 1, m, E)
    for b in range(B):
        qb, kr, vr = bits(x["q"][b]), bits(x["k_raw"][b]), bits(x["v_raw"][b])
        sc = O.f64_to_bf16_rne(O.index_scores(npy(x["qi_codes"][b, 0]), npy(x["qi_scales"][b, 0]),
                                              npy(x["ki_codes"][b]), npy(x["ki_scales"][b]), 64))
        ridx, rcnt = O.topk_select(sc, nv, k)
        assert int(npy(layer["topk_cnt"][b])[0]) == rcnt
        np.testing.assert_array_equal(npy(layer["topk_idx"][b, 0]), ridx, err_msg=f"b={b}")
        o, l = O.csa_attend_one(O.bf16_to_f64(qb[0]), f64(layer["k_cmp"][b]),
                                f64(layer["v_cmp"][b]), ridx, rcnt, O.bf16_to_f64(kr),
                                O.bf16_to_f64(vr), N - 1, W)
        assert_attention_close(f64(layer["out"][b, 0]), o, f"out b={b}")
        assert_lse_close(npy(layer["lse"][b, 0]), l, f"lse b={b}")


@pytest.mark.parametrize("B,N,Nq,H,d", [(2, 8192, 1, 64, 128),    # decode: the one-launch step
                                        (1, 2048, 40, 64, 128),   # prefill rows
                                        (1, 1024, 24, 8, 64)])    # head dim 64, packed prefill
def test_shared_kv_buffers(B, N, Nq, H, d):
    """Shared-KV models pass one buffer as both K and V (raw and pooled): k_raw is v_raw and
    k_cmp is v_cmp. Both layers of a pair must match the oracle run with V = K."""
    m, k, W = 4, 64, 32
    q0 = N - Nq
    cb = (q0 // m) * m if Nq > 1 else N - m
    s = LayerShape("csa", B=B, N=N, Nq=Nq, q_pos0=q0, H=H, d=d, m=m, W=W, k=k, H_I=4, d_I=64,
                   q_scale=1.0 / np.sqrt(d), compress_begin=cb)
    x = generate_layer(s, seed=N + Nq + d, device=DEV)
    kv = x["k_raw"]  # one raw buffer
    E = N // m
    cmp = torch.empty((B, E, d), dtype=torch.bfloat16, device=DEV)  # one pooled buffer
    if cb > 0:
        csa.compress(kv, kv, x["logits"], m, cmp, cmp, 0, cb)
    layer = dict(q=x["q"], k_raw=kv, v_raw=kv, logits=x["logits"], qi_codes=x["qi_codes"],
                 qi_scales=x["qi_scales"], ki_codes=x["ki_codes"], ki_scales=x["ki_scales"],
                 k_cmp=cmp, v_cmp=cmp, out=torch.empty_like(x["q"]),
                 topk_idx=torch.empty((B, Nq, k), dtype=torch.int32, device=DEV),
                 topk_cnt=torch.empty((B, Nq), dtype=torch.int32, device=DEV),
                 m=m, W=W, k=k, q_pos0=q0, compress_begin=cb)
    hs = LayerShape("hca", B=B, N=N, Nq=Nq, q_pos0=q0, H=H, d=d, m=128, W=W, k=0, H_I=0, d_I=0,
                    q_scale=1.0 / np.sqrt(d), compress_begin=(q0 // 128) * 128 if Nq > 1 else N - 128)
    hx = generate_layer(hs, seed=N + 7, device=DEV)
    hkv, hE = hx["k_raw"], N // 128
    hcmp = torch.empty((B, hE, d), dtype=torch.bfloat16, device=DEV)
    if hs.compress_begin > 0:
        csa.compress(hkv, hkv, hx["logits"], 128, hcmp, hcmp, 0, hs.compress_begin)
    hlayer = dict(q=hx["q"], k_raw=hkv, v_raw=hkv, logits=hx["logits"], k_cmp=hcmp, v_cmp=hcmp,
                  out=torch.empty_like(hx["q"]), m=128, W=W, q_pos0=q0,
                  compress_begin=hs.compress_begin)
    csa.layer_pair(layer, hlayer)
    torch.cuda.synchronize()
    assert csa.device_status(reset=True) == 0
    for b in range(B):
        qb, kr = bits(x["q"][b]), bits(kv[b])
        ref = O.csa_layer_seq(qb, kr, kr, npy(x["logits"][b]), npy(x["qi_codes"][b]),
                              npy(x["qi_scales"][b]), npy(x["ki_codes"][b]),
                              npy(x["ki_scales"][b]), m=m, W=W, k=k, d_I=64, q_pos0=q0)
        np.testing.assert_array_equal(npy(layer["topk_idx"][b]), ref["idx"], err_msg=f"b={b}")
        assert_attention_close(f64(layer["out"][b]), ref["out"], f"csa b={b}")
        hr = O.hca_layer_seq(bits(hx["q"][b]), bits(hkv[b]), bits(hkv[b]), npy(hx["logits"][b]),
                             m=128, W=W, q_pos0=q0)
        assert_attention_close(f64(hlayer["out"][b]), hr["out"], f"hca b={b}")
