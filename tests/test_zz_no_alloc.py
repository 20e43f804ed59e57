"""csa_index_topk_noalloc: the indexer + top-k entry point for callers that cannot allocate
device memory (a plugin whose memory belongs to a host framework's pool, code that must avoid
cudaMalloc's implicit synchronisation, a C caller holding only its input and output pointers).
Its score scratch is a fixed array inside the library instead of a workspace.

Called here through the C ABI and compared with the allocating csa_index_topk on two calls in a
row with different inputs, so scratch left over by the first call cannot leak into the second;
the second, smaller call of each pair is also checked against the fp64 oracle's scores and
selection, so a fault shared by both entry points would still show. Top-k lists are integer
results: the comparisons are exact, as for every top-k test. This file is
collected last so a failure here stops a `-x` run only after every other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
from long_context_compressed_pooling_b300 import _native as N
from synth import LayerShape, generate_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, B, Nq, q_pos0, N_ctx, m, H_I, d_I):
    s = LayerShape("csa", B=B, N=N_ctx, Nq=Nq, q_pos0=q_pos0, H=8, d=64, m=m, W=8, k=1,
                   H_I=H_I, d_I=d_I, q_scale=0.125, compress_begin=0)
    return generate_layer(s, seed, device=DEV, skip=("q", "k_raw", "v_raw", "logits"))


def _noalloc(x, q_pos0, m, k):
    lib = N.load_library()
    B, Nq, H_I, half = x["qi_codes"].shape
    E = x["ki_codes"].shape[1]
    idx = torch.full((B, Nq, k), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((B, Nq), -7, dtype=torch.int32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = lib.csa_index_topk_noalloc(
        p(x["qi_codes"]), p(x["qi_scales"]), p(x["ki_codes"]), p(x["ki_scales"]), B, Nq, q_pos0,
        E, m, H_I, 2 * half, k, p(idx), p(cnt),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, csa.load_library().csa_status_string(code)
    return idx, cnt


@pytest.mark.parametrize("first,second", [
    # (seed, B, Nq, q_pos0, N, m, H_I, d_I, k)
    ((21, 16, 1, 131071, 131072, 4, 4, 64, 512), (22, 3, 40, 900, 1000, 4, 2, 32, 24)),
    ((23, 2, 70, 500, 600, 4, 4, 64, 24), (24, 4, 1, 8191, 8192, 4, 8, 64, 300)),
])
def test_noalloc_matches_allocating_entry_point_twice(first, second):
    for call, (seed, B, Nq, q_pos0, N_ctx, m, H_I, d_I, k) in enumerate((first, second)):
        x = _inputs(seed, B, Nq, q_pos0, N_ctx, m, H_I, d_I)
        ref_idx, ref_cnt, _ = csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"],
                                             x["ki_scales"], q_pos0, m, k)
        got_idx, got_cnt = _noalloc(x, q_pos0, m, k)
        torch.cuda.synchronize()
        gi, gc = got_idx.cpu().numpy(), got_cnt.cpu().numpy()
        assert np.array_equal(gc, ref_cnt.cpu().numpy())
        assert np.array_equal(gi, ref_idx.cpu().numpy())
        if call == 1:  # the oracle: exact scores rounded to BF16, then the selection rule
            qc, qs, kc, ks = (x[n].cpu().numpy() for n in ("qi_codes", "qi_scales", "ki_codes",
                                                           "ki_scales"))
            E = N_ctx // m
            for b in range(B):
                for i in range(Nq):
                    nv = O.visible_entries(q_pos0 + i, m, E)
                    sc = O.f64_to_bf16_rne(O.index_scores(qc[b, i], qs[b, i], kc[b, :nv],
                                                          ks[b, :nv], d_I))
                    ridx, rcnt = O.topk_select(sc, nv, k)
                    assert gc[b, i] == rcnt and np.array_equal(gi[b, i], ridx), (b, i)
    assert csa.device_status(reset=True) == 0


def test_noalloc_rejects_more_scores_than_its_scratch():
    lib = N.load_library()
    a = ctypes.c_void_p(0x10000)
    # 2 x 1 x 4,194,304 scores: twice the fixed scratch
    code = lib.csa_index_topk_noalloc(a, a, a, a, 2, 1, 0, 1 << 22, 4, 4, 64, 8, a, a, None)
    assert code == 4  # CSA_ERR_WORKSPACE, returned before anything is launched
