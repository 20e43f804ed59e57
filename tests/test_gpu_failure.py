"""Device-side failure detection, exercised without faulting the GPU.

Every wait of the library's kernels on data another warp or an asynchronous copy produces is
bounded. A test shortens the bound (csa_test_set_faults) and makes the producer of one wait skip
its work, so that the wait runs out: the kernel must record CSA_DEVFLAG_TIMEOUT in the status
word, release what it holds (tensor memory) and return, and the context must stay usable: the
same call without the injected fault afterwards gives the oracle's result."""
import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa
import oracle as O
from synth import LayerShape, generate_layer
from _helpers import bits, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 0x2
BUDGET = 2_000_000  # SM cycles: about 1 ms at 2 GHz


@pytest.fixture(autouse=True)
def _restore():
    if torch.cuda.is_available():
        csa.device_status(reset=True)
    yield
    csa.test_set_faults(0, 0)
    if torch.cuda.is_available():
        csa.device_status(reset=True)


def _check_against_oracle(x, q_pos0, m, k, E, idx, cnt, scb, B, Nq, d_I):
    qc, qs, kc, ks = (npy(x[n]) for n in ("qi_codes", "qi_scales", "ki_codes", "ki_scales"))
    for b in range(B):
        for i in range(Nq):
            nv = O.visible_entries(q_pos0 + i, m, E)
            ref = O.f64_to_bf16_rne(O.index_scores(qc[b, i], qs[b, i], kc[b, :nv], ks[b, :nv], d_I))
            assert np.array_equal(scb[b, i, :nv], ref), (b, i)
            ridx, rcnt = O.topk_select(ref, nv, k)
            assert cnt[b, i] == rcnt and np.array_equal(idx[b, i], ridx), (b, i)


@pytest.mark.parametrize("B,Nq,q_pos0,N,k", [(3, 1, 4095, 4096, 64),     # decode
                                            (1, 40, 2000, 2048, 16)])   # prefill groups
def test_indexer_wait_runs_out_and_the_context_stays_usable(B, Nq, q_pos0, N, k):
    m, H_I, d_I = 4, 4, 64
    s = LayerShape("csa", B=B, N=N, Nq=Nq, q_pos0=q_pos0, H=8, d=64, m=m, W=8, k=k, H_I=H_I,
                   d_I=d_I, q_scale=0.125, compress_begin=0)
    x = generate_layer(s, seed=31 + Nq, device=DEV, skip=("q", "k_raw", "v_raw", "logits"))
    E = N // m
    # the key copies never arrive: the MMA and epilogue waits on them must give up
    csa.test_set_faults(BUDGET, csa.FAULT_SKIP_KEY_COPIES)
    csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"], q_pos0, m, k,
                   want_scores=True)
    flags = csa.device_status(reset=True)
    assert flags & TIMEOUT, f"status {flags:#x}: no wait recorded its expiry"
    # same call, no fault: the kernel left nothing behind (tensor memory freed, barriers unused)
    csa.test_set_faults(0, 0)
    idx, cnt, sc = csa.index_topk(x["qi_codes"], x["qi_scales"], x["ki_codes"], x["ki_scales"],
                                  q_pos0, m, k, want_scores=True)
    assert csa.device_status(reset=True) == 0
    _check_against_oracle(x, q_pos0, m, k, E, npy(idx), npy(cnt), bits(sc), B, Nq, d_I)


def test_unknown_fault_bits_are_refused():
    with pytest.raises(csa.CsaError):
        csa.test_set_faults(0, 0x80)
