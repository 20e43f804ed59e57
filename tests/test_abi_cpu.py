"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports every function
include/csa.h declares, rejects bad arguments before touching CUDA, sizes workspaces, and the
ctypes descriptor structs match the C layout."""
import ctypes
import os

import pytest
import torch

from long_context_compressed_pooling_b300 import build as B
import long_context_compressed_pooling_b300 as csa
from long_context_compressed_pooling_b300 import _native as N


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.load_library()


def test_every_declared_symbol_is_exported(lib):
    syms = N.exported_symbols()
    assert len(syms) >= 14
    missing = [n for n, ok in syms.items() if not ok]
    assert not missing, missing
    assert lib.csa_abi_version() == 3


def test_status_strings(lib):
    for code in range(8):
        s = lib.csa_status_string(code)
        assert s and s != b"unknown status"
    assert lib.csa_status_string(99) == b"unknown status"


def _p(addr):
    return ctypes.c_void_p(addr)


ALN = 0x10000  # fake but aligned device addresses: validation fails before they are used


def test_compress_validation(lib):
    f = lib.csa_compress
    ok = dict(k=_p(ALN), v=_p(ALN), w=_p(ALN), kc=_p(ALN * 2), vc=_p(ALN * 3))
    # null pointer
    assert f(None, ok["v"], ok["w"], 1, 64, 128, 4, 0, 64, ok["kc"], ok["vc"], None) == 1
    # misaligned
    assert f(_p(ALN + 2), ok["v"], ok["w"], 1, 64, 128, 4, 0, 64, ok["kc"], ok["vc"], None) == 3
    # tok_begin not a multiple of m, tok_end beyond N
    assert f(ok["k"], ok["v"], ok["w"], 1, 64, 128, 4, 2, 64, ok["kc"], ok["vc"], None) == 2
    assert f(ok["k"], ok["v"], ok["w"], 1, 64, 128, 4, 0, 65, ok["kc"], ok["vc"], None) == 2
    # unsupported head dim / block size
    assert f(ok["k"], ok["v"], ok["w"], 1, 64, 96, 4, 0, 64, ok["kc"], ok["vc"], None) == 5
    assert f(ok["k"], ok["v"], ok["w"], 1, 64, 128, 3, 0, 63, ok["kc"], ok["vc"], None) == 5
    assert f(ok["k"], ok["v"], ok["w"], 1, 1024, 128, 512, 0, 1024, ok["kc"], ok["vc"], None) == 5
    # shared output cache with distinct K and V inputs
    assert f(ok["k"], _p(ALN * 5), ok["w"], 1, 64, 128, 4, 0, 64, ok["kc"], ok["kc"], None) == 1


def test_index_and_attend_validation(lib):
    a = _p(ALN)
    f = lib.csa_index_topk
    # unsupported d_I and H_I
    assert f(a, a, a, a, 1, 1, 0, 16, 4, 4, 48, 8, a, a, None, None, 0, None) == 5
    assert f(a, a, a, a, 1, 1, 0, 16, 4, 3, 64, 8, a, a, None, None, 0, None) == 5
    # k = 0
    assert f(a, a, a, a, 1, 1, 0, 16, 4, 4, 64, 0, a, a, None, None, 0, None) == 1
    # no scores buffer and no workspace
    assert f(a, a, a, a, 1, 1, 0, 16, 4, 4, 64, 8, a, a, None, None, 0, None) == 4
    g = lib.csa_attend
    # queries beyond the context
    assert g(a, a, a, 4, a, a, 2, a, a, 10, 4, 1, 2, 9, 8, 64, a, None, None, 0, None) == 2
    # unsupported head dim
    assert g(a, a, a, 4, a, a, 2, a, a, 10, 4, 1, 1, 9, 8, 96, a, None, None, 0, None) == 5
    h = lib.hca_attend
    assert h(a, a, a, 4, 0, a, a, 10, 4, 1, 1, 9, 8, 64, a, None, None, 0, None) == 1
    assert lib.csa_hca_layer_pair(None, None, None, 0, None) == 1


def test_workspace_sizes(lib):
    # prefill-sized attention needs no split-K workspace; small decode batches do
    assert lib.csa_attend_workspace_size(1, 8192, 64, 128, 2048, 128) == 0
    ws = lib.csa_attend_workspace_size(16, 1, 64, 128, 512, 128)
    assert ws > 0 and ws % 4 == 0
    assert lib.hca_attend_workspace_size(32, 1, 64, 128, 8192, 128, 128) > 0
    # scores live in the workspace unless the caller passes a buffer
    assert lib.csa_index_topk_workspace_size(16, 1, 32768, 512, 0) >= 16 * 32768 * 2
    assert lib.csa_index_topk_workspace_size(16, 1, 32768, 512, 1) == 0


def test_index_key_and_quantizer_validation(lib):
    f = lib.csa_compress_index_keys
    x, w, c, sc = _p(ALN), _p(ALN * 2), _p(ALN * 3), _p(ALN * 4)
    assert f(None, w, 1, 64, 64, 4, 0, 64, c, sc, None) == 1          # null pointer
    assert f(_p(ALN + 2), w, 1, 64, 64, 4, 0, 64, c, sc, None) == 3   # misaligned rows
    assert f(x, w, 1, 64, 64, 4, 2, 64, c, sc, None) == 2             # tok_begin % m
    assert f(x, w, 1, 64, 64, 4, 0, 65, c, sc, None) == 2             # tok_end > N
    assert f(x, w, 1, 64, 48, 4, 0, 64, c, sc, None) == 5             # d_I
    assert f(x, w, 1, 128, 64, 64, 0, 128, c, sc, None) == 5          # m > 32
    assert f(x, w, 1, 64, 64, 3, 0, 63, c, sc, None) == 5             # m not a power of two
    q = lib.csa_quantize_mxfp4
    assert q(None, 4, 64, c, sc, None) == 1
    assert q(x, 4, 64, _p(ALN + 1), sc, None) == 3
    assert q(x, -1, 64, c, sc, None) == 2
    assert q(x, 4, 96, c, sc, None) == 5


def test_fp32_score_path_validation(lib):
    f = lib.csa_topk_f32
    s_, i_, c_ = _p(ALN), _p(ALN * 2), _p(ALN * 3)
    assert f(None, 1, 1, 0, 100, 4, 8, i_, c_, None) == 1
    assert f(_p(ALN + 4), 1, 1, 0, 100, 4, 8, i_, c_, None) == 3
    assert f(s_, 1, 1, 0, 100, 4, 0, i_, c_, None) == 1              # k < 1
    # rows above 16 x 32768 visible entries are not implemented for FP32 scores
    assert f(s_, 1, 1, 4 * 600000 - 1, 600000, 4, 8, i_, c_, None) == 5
    g = lib.csa_index_scores
    a = _p(ALN)
    assert g(a, a, a, a, 1, 1, 0, 100, 4, 4, 64, None, None, None) == 1    # no BF16 buffer
    assert g(a, a, a, a, 1, 1, 0, 100, 4, 4, 64, a, _p(ALN + 8), None) == 3
    assert g(a, a, a, a, 1, 1, 0, 100, 4, 4, 48, a, None, None) == 5


def _paged(**kw):
    d = N.PagedLayerDesc()
    d.kind, d.B, d.H, d.d, d.m, d.W, d.k, d.H_I, d.d_I = 0, 2, 64, 128, 4, 128, 64, 4, 64
    d.N, d.n_pages, d.max_blocks = 5000, 8, 2
    for f in ("k_pool", "v_pool", "ki_codes_pool", "ki_scales_pool", "block_table", "ring_k",
              "ring_v", "ring_logits", "k_new", "v_new", "logit_new", "q", "qi_codes",
              "qi_scales", "out", "topk_idx", "topk_cnt"):
        setattr(d, f, ALN)
    for k, v in kw.items():
        setattr(d, k, v)
    return ctypes.pointer(d)


def test_paged_validation(lib):
    f = lambda **kw: lib.csa_paged_decode_step(_paged(**kw), None, 0, None)
    assert f(kind=2) == 1
    assert f(q=None) == 1
    assert f(ring_xi=ALN) == 1                 # index-key rows in the ring but no new row
    assert f(k_pool=ALN + 8) == 3
    assert f(N=3 * 4096) == 2                  # the appended token beyond the block table
    assert f(W=200) == 5
    assert f(m=64) == 5                        # CSA pages must hold whole indexer tiles
    assert f(d_I=32) == 5
    assert f(kind=1, m=256) == 5
    assert f() == 4                            # valid descriptor, no workspace
    assert lib.csa_paged_decode_workspace_size(_paged()) > 0
    assert lib.csa_paged_decode_workspace_size(_paged(kind=2)) == 0
    # the pair takes a CSA layer then an HCA layer
    g = lib.csa_paged_layer_pair
    hca = _paged(kind=1, m=128, k=0)
    assert g(_paged(), _paged(), None, 0, None) == 1
    assert g(hca, _paged(), None, 0, None) == 1
    assert g(_paged(), None, None, 0, None) == 1
    assert g(_paged(), _paged(kind=1, m=256), None, 0, None) == 5
    assert g(_paged(), hca, None, 0, None) == 4
    both = lib.csa_paged_layer_pair_workspace_size(_paged(), hca)
    assert both >= lib.csa_paged_decode_workspace_size(_paged()) + \
        lib.csa_paged_decode_workspace_size(hca)


def test_descriptor_struct_layout():
    # 15 pointers, 9 ints (+4 padding), 3 int64, 1 pointer / 8 pointers, 6 ints, 3 int64
    assert ctypes.sizeof(N.CsaLayerDesc) == 15 * 8 + 9 * 4 + 4 + 3 * 8 + 8
    assert N.CsaLayerDesc.N.offset == 160
    assert N.CsaLayerDesc.xi_raw.offset == 184
    assert ctypes.sizeof(N.HcaLayerDesc) == 8 * 8 + 6 * 4 + 3 * 8
    assert N.HcaLayerDesc.N.offset == 88
    # 9 ints (+4 padding), int64, 5 pointers, 2 ints, 15 pointers
    assert ctypes.sizeof(N.PagedLayerDesc) == 9 * 4 + 4 + 8 + 5 * 8 + 2 * 4 + 15 * 8
    assert N.PagedLayerDesc.N.offset == 40 and N.PagedLayerDesc.ring_k.offset == 96


def test_library_is_sm103a_build():
    # the build targets sm_103a only
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.ARCH)
    assert os.path.exists(N.LIB_PATH)


def test_missing_library_raises(monkeypatch, tmp_path):
    """No fallback: without the library the first call raises instead of computing anything."""
    monkeypatch.setattr(N, "_lib", None)
    monkeypatch.setattr(N, "LIB_PATH", str(tmp_path / "libcsa_b300.so"))
    with pytest.raises(RuntimeError, match="is missing"):
        N.load_library()
    with pytest.raises(RuntimeError, match="is missing"):
        csa.topk(torch.zeros((1, 1, 8), dtype=torch.bfloat16), 7, 1, 2)


def test_host_tensors_are_refused(lib):
    """Host tensors never reach a computation: the binding rejects them before any call."""
    s = torch.zeros((1, 1, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA device"):
        csa.topk(s, 7, 1, 2)
    with pytest.raises(ValueError, match="CUDA device"):
        csa.topk_f32(s.float(), 7, 1, 2)
    with pytest.raises(ValueError, match="CUDA device"):
        csa.quantize_mxfp4(torch.zeros((4, 64), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA device"):
        z = torch.zeros((2, 8), dtype=torch.bfloat16)
        csa.scatter_rows([(z, z.clone())])


def test_fault_injection_switches_are_validated_and_restorable(lib):
    # host-only: the switches are stored for later launches, nothing touches CUDA here
    assert lib.csa_test_set_faults(1000, 0x80) == 1   # unknown producer bit
    assert lib.csa_test_set_faults(2_000_000, 0x1) == 0
    assert lib.csa_test_set_faults(0, 0) == 0          # defaults restored


def test_sharded_calls_validate_before_launching(lib):
    a = _p(ALN)
    bases = (ctypes.c_int64 * 3)(0, 100, 50)  # not ascending
    assert lib.csa_topk_merge(a, a, a, bases, 2, 3, 64, a, a, a, a, None) == 2
    ok = (ctypes.c_int64 * 17)(*range(0, 1700, 100))
    assert lib.csa_topk_merge(a, a, a, ok, 2, 17, 64, a, a, a, a, None) == 5   # S > 16
    assert lib.csa_topk_merge(a, a, a, ok, 2, 4, 4096, a, a, a, a, None) == 5  # k > 2048
    assert lib.csa_topk_merge(None, a, a, ok, 2, 4, 64, a, a, a, a, None) == 1
    assert lib.csa_lse_merge(a, a, 2, 10, 60, a, None, None) == 5              # d % 8
    assert lib.csa_lse_merge(a, a, 0, 10, 64, a, None, None) == 1
    assert lib.csa_shard_candidates_workspace_size(2, 1000, 64) == 4096


def test_scatter_rows_validates_before_launching(lib):
    # host-only: every refused call returns before touching CUDA; copies that move no byte are
    # dropped, so a call made of them launches nothing
    a = _p(ALN)
    D = N.CopyDesc
    assert lib.csa_scatter_rows(None, 1, None) == 1                    # no descriptors
    assert lib.csa_scatter_rows((D * 1)(), -1, None) == 1              # negative count
    assert lib.csa_scatter_rows((D * 17)(), 17, None) == 1             # above CSA_MAX_COPIES
    assert lib.csa_scatter_rows((D * 1)(D(a, a, -1, 16, 16)), 1, None) == 1   # negative rows
    assert lib.csa_scatter_rows((D * 1)(D(a, a, 2, 32, 16)), 1, None) == 1    # stride < row
    assert lib.csa_scatter_rows((D * 1)(D(None, a, 2, 16, 16)), 1, None) == 1  # null dst
    assert lib.csa_scatter_rows((D * 2)(D(None, None, 0, 16, 16), D(None, None, 3, 0, 0)), 2,
                                None) == 0                             # nothing to move
    assert lib.csa_scatter_rows(None, 0, None) == 0
