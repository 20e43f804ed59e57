"""The paged heterogeneous KV cache with incremental decode-time compression, against the fp64
oracle on the logical sequence.

A prefix is placed in pages (mapped through a shuffled block table) and in the 256-token rings;
then tokens are decoded one by one with csa_paged_decode_step, each call appending its token and
compressing the block it closes. Every step's top-k is compared bit for bit and its output within
the attention tolerance with the oracle's decode of the same logical sequence at that position;
afterwards the entries the calls wrote into the pages are compared with the oracle's pooling
and the rings with the raw rows. The steps cross a page boundary and close CSA and HCA blocks."""
import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
from synth import LayerShape, generate_layer, index_key_rows
from _helpers import assert_attention_close, assert_entries_close, bits, f64, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"
P, R = csa.PAGE_TOKENS, csa.RING_TOKENS


@pytest.fixture(autouse=True)
def _clean_status():
    if torch.cuda.is_available():
        csa.device_status(reset=True)
    yield
    if torch.cuda.is_available():
        assert csa.device_status(reset=True) == 0


def _layout(B, n_blocks, spare, seed):
    """Pages of every (sequence, block) in a shuffled order, plus unused spare pages."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(B * n_blocks + spare)[: B * n_blocks].reshape(B, n_blocks)
    return torch.from_numpy(perm.astype(np.int32)).to(DEV), B * n_blocks + spare


def _to_pages(flat, table, n_pages, per_page):
    """Scatter flat per-sequence rows [B, E, ...] into pool pages (test set-up)."""
    B, E = flat.shape[:2]
    pool = torch.zeros((n_pages, per_page) + tuple(flat.shape[2:]), dtype=flat.dtype, device=DEV)
    for b in range(B):
        for j0 in range(0, E, per_page):
            n = min(per_page, E - j0)
            pool[int(table[b, j0 // per_page]), :n] = flat[b, j0:j0 + n]
    return pool


def _from_pages(pool, table, b, j0, j1, per_page):
    rows = [pool[int(table[b, j // per_page]), j % per_page] for j in range(j0, j1)]
    return torch.stack(rows)


def _rings(x, d_key, N0):
    """Rings holding the raw rows of positions max(0, N0 - 256) .. N0 - 1."""
    B = x.shape[0]
    ring = torch.zeros((B, R) + tuple(x.shape[2:]), dtype=x.dtype, device=DEV)
    for pos in range(max(0, N0 - R), N0):
        ring[:, pos % R] = x[:, pos]
    return ring


def _setup(kind, B, N0, T, m, W, k, seed, xi_rows):
    H, d, H_I, d_I = 64, 128, 4, 64
    N = N0 + T
    s = LayerShape(kind, B=B, N=N, Nq=T, q_pos0=N0, H=H, d=d, m=m, W=W, k=k, H_I=H_I,
                   d_I=d_I, q_scale=1.0 / np.sqrt(d), compress_begin=0)
    x = generate_layer(s, seed=seed, device=DEV)
    n_blocks = (N + P - 1) // P
    table, n_pages = _layout(B, n_blocks, 3, seed)
    per_page = P // m
    E0 = N0 // m
    kc = torch.empty((B, E0, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    csa.compress(x["k_raw"][:, :N0].contiguous(), x["v_raw"][:, :N0].contiguous(),
                 x["logits"][:, :N0].contiguous(), m, kc, vc)
    L = dict(kind=kind, m=m, W=W, k=k, N=N0, block_table=table,
             k_pool=_to_pages(kc, table, n_pages, per_page),
             v_pool=_to_pages(vc, table, n_pages, per_page),
             ring_k=_rings(x["k_raw"], d, N0), ring_v=_rings(x["v_raw"], d, N0),
             ring_logits=_rings(x["logits"], 1, N0),
             out=torch.empty((B, H, d), dtype=torch.bfloat16, device=DEV))
    xi = None
    if kind == "csa":
        if xi_rows:
            xi = index_key_rows(s, seed=seed, device=DEV)
            c0, s0 = csa.compress_index_keys(xi[:, :N0].contiguous(), x["logits"][:, :N0].contiguous(), m)
            L["ring_xi"] = _rings(xi, d_I, N0)
        else:  # the keys of every entry the steps will reach are inputs, already in the pages
            c0, s0 = x["ki_codes"], x["ki_scales"]
        L["ki_codes_pool"] = _to_pages(c0, table, n_pages, per_page)
        L["ki_scales_pool"] = _to_pages(s0, table, n_pages, per_page)
        L["topk_idx"] = torch.empty((B, k), dtype=torch.int32, device=DEV)
        L["topk_cnt"] = torch.empty((B,), dtype=torch.int32, device=DEV)
    return s, x, xi, L


def _run_steps(s, x, xi, L, T, check):
    for i in range(T):
        t = s.q_pos0 + i
        L.update(N=t, k_new=x["k_raw"][:, t].contiguous(), v_new=x["v_raw"][:, t].contiguous(),
                 logit_new=x["logits"][:, t].contiguous(), q=x["q"][:, i].contiguous())
        if s.kind == "csa":
            L.update(qi_codes=x["qi_codes"][:, i].contiguous(),
                     qi_scales=x["qi_scales"][:, i].contiguous())
            if xi is not None:
                L["xi_new"] = xi[:, t].contiguous()
        csa.paged_decode_step(L)
        torch.cuda.synchronize()
        assert csa.device_status(reset=True) == 0, f"step {i}"
        check(i, t)


@pytest.mark.parametrize("B,N0,T,k", [(2, 2 * P - 6, 12, 64),   # crosses the page boundary
                                      (1, 300, 9, 512)])        # short context, k > visible
def test_paged_csa_decode_matches_oracle(B, N0, T, k):
    m, W = 4, 128
    s, x, _, L = _setup("csa", B, N0, T, m, W, k, seed=N0 + T, xi_rows=False)
    qb, kr, vr = bits(x["q"]), bits(x["k_raw"]), bits(x["v_raw"])

    def check(i, t):
        idx, cnt, out = npy(L["topk_idx"]), npy(L["topk_cnt"]), L["out"]
        for b in range(B):
            ref = O.csa_layer_seq(qb[b], kr[b], vr[b], npy(x["logits"][b]),
                                  npy(x["qi_codes"][b]), npy(x["qi_scales"][b]),
                                  npy(x["ki_codes"][b]), npy(x["ki_scales"][b]), m=m, W=W, k=k,
                                  d_I=64, q_pos0=s.q_pos0, query_rows=[i])
            assert int(cnt[b]) == int(ref["cnt"][0]), (i, b)
            np.testing.assert_array_equal(idx[b], ref["idx"][0], err_msg=f"step {i} b={b}")
            assert_attention_close(f64(out[b]), ref["out"][0], f"step {i} b={b}")

    _run_steps(s, x, None, L, T, check)
    # the entries the steps closed, read back through the block table, and the rings
    j0, j1 = N0 // m, (N0 + T) // m
    for b in range(B):
        ref_k = O.compress(O.bf16_to_f64(kr[b]), npy(x["logits"][b]).astype(np.float64), m)
        ref_v = O.compress(O.bf16_to_f64(vr[b]), npy(x["logits"][b]).astype(np.float64), m)
        assert_entries_close(bits(_from_pages(L["k_pool"], L["block_table"], b, j0, j1, P // m)),
                             ref_k[j0:j1], f"K entries b={b}")
        assert_entries_close(bits(_from_pages(L["v_pool"], L["block_table"], b, j0, j1, P // m)),
                             ref_v[j0:j1], f"V entries b={b}")
        for pos in range(max(0, N0 + T - R), N0 + T):
            assert torch.equal(L["ring_k"][b, pos % R], x["k_raw"][b, pos])


@pytest.mark.parametrize("N0,T", [(2 * P - 3, 6),   # closes HCA block 63 at the page's last token
                                  (130, 4)])        # early context: one entry visible
def test_paged_hca_decode_matches_oracle(N0, T):
    B, m, W = 2, 128, 128
    s, x, _, L = _setup("hca", B, N0, T, m, W, 0, seed=N0, xi_rows=False)
    qb, kr, vr = bits(x["q"]), bits(x["k_raw"]), bits(x["v_raw"])

    def check(i, t):
        for b in range(B):
            ref = O.hca_layer_seq(qb[b], kr[b], vr[b], npy(x["logits"][b]), m=m, W=W,
                                  q_pos0=s.q_pos0, query_rows=[i])
            assert_attention_close(f64(L["out"][b]), ref["out"][0], f"step {i} b={b}")

    _run_steps(s, x, None, L, T, check)
    j0, j1 = N0 // m, (N0 + T) // m
    for b in range(B if j1 > j0 else 0):  # the entries the steps closed, if any
        ref_k = O.compress(O.bf16_to_f64(kr[b]), npy(x["logits"][b]).astype(np.float64), m)
        got = _from_pages(L["k_pool"], L["block_table"], b, j0, j1, P // m)
        assert_entries_close(bits(got), ref_k[j0:j1], f"HCA entries b={b}")


def test_paged_steps_pool_their_index_keys():
    """With index-key rows in the state cache, the steps write the keys of the entries they close
    (MX FP4, as csa_compress_index_keys); they match the oracle as in test_gpu_index_keys, and
    equal the standalone conversion of the whole sequence bit for bit."""
    from test_gpu_index_keys import _check_seq_keys
    B, N0, T, m, k = 2, P - 5, 10, 4, 64
    s, x, xi, L = _setup("csa", B, N0, T, m, 128, k, seed=5, xi_rows=True)
    _run_steps(s, x, xi, L, T, lambda i, t: None)
    full_c, full_s = csa.compress_index_keys(xi, x["logits"], m)
    j0, j1 = N0 // m, (N0 + T) // m
    for b in range(B):
        gc = _from_pages(L["ki_codes_pool"], L["block_table"], b, j0, j1, P // m)
        gs = _from_pages(L["ki_scales_pool"], L["block_table"], b, j0, j1, P // m)
        assert torch.equal(gc, full_c[b, j0:j1]) and torch.equal(gs, full_s[b, j0:j1])
        codes = np.zeros((j1, 32), np.uint8)
        scales = np.zeros((j1, 2), np.uint8)
        codes[j0:j1], scales[j0:j1] = npy(gc), npy(gs)
        _check_seq_keys(codes, scales, bits(xi[b, :j1 * m]), npy(x["logits"][b, :j1 * m]), m,
                        j0, j1, f"paged b={b}")


def test_unmapped_page_is_flagged_not_faulted():
    """A block-table entry outside the pool is an input error: the call flags it in the device
    status word and leaves those keys out; nothing outside the pools is touched."""
    B, N0, k = 1, P + 100, 32
    s, x, _, L = _setup("csa", B, N0, 1, 4, 128, k, seed=9, xi_rows=False)
    L["block_table"][0, 0] = L["k_pool"].shape[0] + 7  # tokens 0..4095 now unmapped
    L.update(N=N0, k_new=x["k_raw"][:, N0].contiguous(), v_new=x["v_raw"][:, N0].contiguous(),
             logit_new=x["logits"][:, N0].contiguous(), q=x["q"][:, 0].contiguous(),
             qi_codes=x["qi_codes"][:, 0].contiguous(), qi_scales=x["qi_scales"][:, 0].contiguous())
    csa.paged_decode_step(L)
    torch.cuda.synchronize()
    assert csa.device_status(reset=True) != 0
    assert torch.isfinite(L["out"].float()).all()


def test_paged_layer_pair_matches_oracle():
    """csa_paged_layer_pair: a CSA and an HCA layer (independent inputs) stepped together, the
    HCA layer on the side stream; both outputs against the oracle at every step."""
    B, N0, T = 2, P - 2, 4
    sc, xc, _, Lc = _setup("csa", B, N0, T, 4, 128, 64, seed=21, xi_rows=False)
    sh, xh, _, Lh = _setup("hca", B, N0, T, 128, 128, 0, seed=22, xi_rows=False)
    for i in range(T):
        t = N0 + i
        for s, x, L in ((sc, xc, Lc), (sh, xh, Lh)):
            L.update(N=t, k_new=x["k_raw"][:, t].contiguous(), v_new=x["v_raw"][:, t].contiguous(),
                     logit_new=x["logits"][:, t].contiguous(), q=x["q"][:, i].contiguous())
        Lc.update(qi_codes=xc["qi_codes"][:, i].contiguous(),
                  qi_scales=xc["qi_scales"][:, i].contiguous())
        csa.PreparedPagedPair(Lc, Lh)()
        torch.cuda.synchronize()
        assert csa.device_status(reset=True) == 0
        for b in range(B):
            rc = O.csa_layer_seq(bits(xc["q"][b]), bits(xc["k_raw"][b]), bits(xc["v_raw"][b]),
                                 npy(xc["logits"][b]), npy(xc["qi_codes"][b]),
                                 npy(xc["qi_scales"][b]), npy(xc["ki_codes"][b]),
                                 npy(xc["ki_scales"][b]), m=4, W=128, k=64, d_I=64, q_pos0=N0,
                                 query_rows=[i])
            np.testing.assert_array_equal(npy(Lc["topk_idx"][b]), rc["idx"][0])
            assert_attention_close(f64(Lc["out"][b]), rc["out"][0], f"CSA step {i} b={b}")
            rh = O.hca_layer_seq(bits(xh["q"][b]), bits(xh["k_raw"][b]), bits(xh["v_raw"][b]),
                                 npy(xh["logits"][b]), m=128, W=128, q_pos0=N0, query_rows=[i])
            assert_attention_close(f64(Lh["out"][b]), rh["out"][0], f"HCA step {i} b={b}")
