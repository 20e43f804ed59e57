"""ctypes binding of libcsa_b300.so (C ABI in include/csa.h).

Argument marshalling only: tensors become device pointers and sizes, torch's current stream
becomes the cudaStream_t, workspaces are torch allocations sized by the library's own
*_workspace_size() calls. Nothing here computes any part of the method.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, Optional, Tuple

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libcsa_b300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "csa.h")

CSA_OK = 0
_STATUS = {0: "ok", 1: "invalid argument", 2: "inconsistent shape", 3: "pointer not 16-byte aligned",
           4: "workspace missing or too small", 5: "unsupported shape", 6: "CUDA error",
           7: "device-side fault recorded"}


class CsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {_STATUS.get(code, 'unknown')} (status {code})")
        self.code = code


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_Z = ctypes.c_size_t


class CsaLayerDesc(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("q", "k_raw", "v_raw", "logits", "qi_codes", "qi_scales",
                                  "ki_codes", "ki_scales", "k_cmp", "v_cmp", "out", "lse",
                                  "topk_idx", "topk_cnt", "scores")] + \
               [(n, _I) for n in ("B", "Nq", "H", "d", "m", "W", "k", "H_I", "d_I")] + \
               [(n, _L) for n in ("N", "q_pos0", "compress_begin")] + [("xi_raw", _P)]


class HcaLayerDesc(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("q", "k_raw", "v_raw", "logits", "k_cmp", "v_cmp", "out",
                                  "lse")] + \
               [(n, _I) for n in ("B", "Nq", "H", "d", "m", "W")] + \
               [(n, _L) for n in ("N", "q_pos0", "compress_begin")]


class PagedLayerDesc(ctypes.Structure):
    _fields_ = [(n, _I) for n in ("kind", "B", "H", "d", "m", "W", "k", "H_I", "d_I")] + \
               [("N", _L)] + \
               [(n, _P) for n in ("k_pool", "v_pool", "ki_codes_pool", "ki_scales_pool",
                                  "block_table")] + \
               [(n, _I) for n in ("n_pages", "max_blocks")] + \
               [(n, _P) for n in ("ring_k", "ring_v", "ring_logits", "ring_xi", "k_new", "v_new",
                                  "logit_new", "xi_new", "q", "qi_codes", "qi_scales", "out",
                                  "lse", "topk_idx", "topk_cnt")]


PAGE_TOKENS = 4096
RING_TOKENS = 256


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", _I), ("total_ms", ctypes.c_double)]


class CopyDesc(ctypes.Structure):
    _fields_ = [("dst", _P), ("src", _P), ("rows", _L), ("row_bytes", _L), ("dst_stride", _L)]


MAX_COPIES = 16


_SIGS = {
    "csa_profiler_enable": (_I, [_I]),
    "csa_profiler_collect": (_I, [ctypes.POINTER(KernelTime), _I, ctypes.POINTER(_I), _I]),
    "csa_compress": (_I, [_P, _P, _P, _I, _L, _I, _I, _L, _L, _P, _P, _P]),
    "csa_compress_index_keys": (_I, [_P, _P, _I, _L, _I, _I, _L, _L, _P, _P, _P]),
    "csa_quantize_mxfp4": (_I, [_P, _L, _I, _P, _P, _P]),
    "csa_index_topk": (_I, [_P, _P, _P, _P, _I, _I, _L, _L, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "csa_index_topk_workspace_size": (_Z, [_I, _I, _L, _I, _I]),
    "csa_index_topk_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _L, _L, _I, _I, _I, _I, _P, _P, _P]),
    "csa_index_scores": (_I, [_P, _P, _P, _P, _I, _I, _L, _L, _I, _I, _I, _P, _P, _P]),
    "csa_topk_f32": (_I, [_P, _I, _I, _L, _L, _I, _I, _P, _P, _P]),
    "csa_topk": (_I, [_P, _I, _I, _L, _L, _I, _I, _P, _P, _P, _Z, _P]),
    "csa_topk_workspace_size": (_Z, [_I, _I, _L, _I]),
    "csa_attend": (_I, [_P, _P, _P, _L, _P, _P, _I, _P, _P, _L, _I, _I, _I, _L, _I, _I, _P, _P, _P,
                        _Z, _P]),
    "csa_attend_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "hca_attend": (_I, [_P, _P, _P, _L, _I, _P, _P, _L, _I, _I, _I, _L, _I, _I, _P, _P, _P, _Z, _P]),
    "hca_attend_workspace_size": (_Z, [_I, _I, _I, _I, _L, _I, _I]),
    "csa_hca_layer_pair": (_I, [ctypes.POINTER(CsaLayerDesc), ctypes.POINTER(HcaLayerDesc), _P, _Z, _P]),
    "csa_hca_layer_pair_workspace_size": (_Z, [ctypes.POINTER(CsaLayerDesc),
                                               ctypes.POINTER(HcaLayerDesc)]),
    "csa_paged_decode_step": (_I, [ctypes.POINTER(PagedLayerDesc), _P, _Z, _P]),
    "csa_paged_decode_workspace_size": (_Z, [ctypes.POINTER(PagedLayerDesc)]),
    "csa_paged_layer_pair": (_I, [ctypes.POINTER(PagedLayerDesc), ctypes.POINTER(PagedLayerDesc),
                                  _P, _Z, _P]),
    "csa_paged_layer_pair_workspace_size": (_Z, [ctypes.POINTER(PagedLayerDesc),
                                                 ctypes.POINTER(PagedLayerDesc)]),
    "csa_get_device_status": (_I, [_P, _I, ctypes.POINTER(ctypes.c_uint32)]),
    "csa_status_string": (ctypes.c_char_p, [_I]),
    "csa_abi_version": (_I, []),
    "csa_test_set_faults": (_I, [ctypes.c_longlong, ctypes.c_uint32]),
    "csa_shard_candidates": (_I, [_P, _P, _P, _P, _I, _L, _L, _I, _I, _I, _I, _P, _P, _P, _P, _Z,
                                  _P]),
    "csa_shard_candidates_workspace_size": (_Z, [_I, _L, _I]),
    "csa_topk_merge": (_I, [_P, _P, _P, ctypes.POINTER(ctypes.c_int64), _I, _I, _I, _P, _P, _P,
                            _P, _P]),
    "csa_lse_merge": (_I, [_P, _P, _I, _L, _I, _P, _P, _P]),
    "csa_scatter_rows": (_I, [ctypes.POINTER(CopyDesc), _I, _P]),
}

_lib: Optional[ctypes.CDLL] = None


def load_library() -> ctypes.CDLL:
    """Load libcsa_b300.so; raise if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m long_context_compressed_pooling_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    """Function names declared in include/csa.h and whether the library exports each."""
    with open(HEADER, encoding="utf-8") as fh:
        text = fh.read()
    names = re.findall(r"^\s*(?:csa_status|size_t|const char\*|int)\s+(\w+)\s*\(", text, re.M)
    lib = load_library()
    return {n: hasattr(lib, n) for n in names}


def _check(fn: str, code: int) -> None:
    if code != CSA_OK:
        raise CsaError(fn, code)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(dev) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ws(nbytes: int, dev, ws: Optional[torch.Tensor]) -> Tuple[Optional[torch.Tensor], int]:
    if nbytes == 0:
        return ws, (ws.numel() if ws is not None else 0)
    if ws is not None and ws.numel() >= nbytes:
        return ws, ws.numel()
    t = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    return t, nbytes


def _u16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("bf16 tensors are expected")
    return t


# ----------------------------------------------------------------------------------------------
def compress(k_raw, v_raw, logits, m: int, k_cmp, v_cmp, tok_begin: int = 0,
             tok_end: Optional[int] = None) -> None:
    """Pool the blocks of tokens [tok_begin, tok_end) into k_cmp / v_cmp ([B, N/m, d])."""
    lib = load_library()
    B, N, d = k_raw.shape
    tok_end = N if tok_end is None else tok_end
    _check("csa_compress", lib.csa_compress(
        _ptr(_u16(k_raw)), _ptr(_u16(v_raw)), _ptr(logits), B, N, d, m, tok_begin, tok_end,
        _ptr(_u16(k_cmp)), _ptr(_u16(v_cmp)), _stream(k_raw.device)))


def compress_index_keys(xi_raw, logits, m: int, ki_codes=None, ki_scales=None,
                        tok_begin: int = 0, tok_end: Optional[int] = None):
    """The indexer's own compressed keys: pool the index-key rows xi_raw [B, N, d_I] (bf16) of
    the blocks in [tok_begin, tok_end) and convert them to MX FP4. Returns (ki_codes
    [B, N/m, d_I/2] uint8, ki_scales [B, N/m, d_I/32] uint8); given buffers are written in
    place (entries outside the range are left untouched)."""
    lib = load_library()
    B, N, d_I = xi_raw.shape
    E = N // m
    dev = xi_raw.device
    if ki_codes is None:
        ki_codes = torch.zeros((B, E, d_I // 2), dtype=torch.uint8, device=dev)
    if ki_scales is None:
        ki_scales = torch.zeros((B, E, d_I // 32), dtype=torch.uint8, device=dev)
    tok_end = N if tok_end is None else tok_end
    _check("csa_compress_index_keys", lib.csa_compress_index_keys(
        _ptr(_u16(xi_raw)), _ptr(logits), B, N, d_I, m, tok_begin, tok_end, _ptr(ki_codes),
        _ptr(ki_scales), _stream(dev)))
    return ki_codes, ki_scales


def quantize_mxfp4(x, codes=None, scales=None):
    """MX FP4 conversion of bf16 rows x [..., d]. Returns (codes [..., d/2] uint8, scales
    [..., d/32] uint8)."""
    lib = load_library()
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    if codes is None:
        codes = torch.empty(x.shape[:-1] + (d // 2,), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (d // 32,), dtype=torch.uint8, device=x.device)
    _check("csa_quantize_mxfp4", lib.csa_quantize_mxfp4(
        _ptr(_u16(x)), rows, d, _ptr(codes), _ptr(scales), _stream(x.device)))
    return codes, scales


def index_topk(qi_codes, qi_scales, ki_codes, ki_scales, q_pos0: int, m: int, k: int,
               topk_idx=None, topk_cnt=None, scores=None, want_scores: bool = False,
               ws: Optional[torch.Tensor] = None):
    """Indexer scores + top-k. Returns (topk_idx [B,Nq,k] int32, topk_cnt [B,Nq] int32, scores
    [B,Nq,E] bf16 or None)."""
    lib = load_library()
    B, Nq, H_I, half = qi_codes.shape
    d_I = 2 * half
    E = ki_codes.shape[1]
    dev = qi_codes.device
    if topk_idx is None:
        topk_idx = torch.empty((B, Nq, k), dtype=torch.int32, device=dev)
    if topk_cnt is None:
        topk_cnt = torch.empty((B, Nq), dtype=torch.int32, device=dev)
    if want_scores and scores is None:
        scores = torch.zeros((B, Nq, E), dtype=torch.bfloat16, device=dev)
    need = lib.csa_index_topk_workspace_size(B, Nq, E, k, 1 if scores is not None else 0)
    ws, wsb = _ws(need, dev, ws)
    _check("csa_index_topk", lib.csa_index_topk(
        _ptr(qi_codes), _ptr(qi_scales), _ptr(ki_codes), _ptr(ki_scales), B, Nq, q_pos0, E, m,
        H_I, d_I, k, _ptr(topk_idx), _ptr(topk_cnt), _ptr(scores), _ptr(ws), wsb,
        _stream(dev)))
    return topk_idx, topk_cnt, scores


def index_scores(qi_codes, qi_scales, ki_codes, ki_scales, q_pos0: int, m: int,
                 want_f32: bool = True, scores=None, scores_f32=None):
    """The indexer alone. Returns (BF16 scores [B,Nq,E], FP32 scores [B,Nq,E] or None); only
    visible entries are written (the rest of freshly allocated buffers is zero)."""
    lib = load_library()
    B, Nq, H_I, half = qi_codes.shape
    E = ki_codes.shape[1]
    dev = qi_codes.device
    if scores is None:
        scores = torch.zeros((B, Nq, E), dtype=torch.bfloat16, device=dev)
    if want_f32 and scores_f32 is None:
        scores_f32 = torch.zeros((B, Nq, E), dtype=torch.float32, device=dev)
    _check("csa_index_scores", lib.csa_index_scores(
        _ptr(qi_codes), _ptr(qi_scales), _ptr(ki_codes), _ptr(ki_scales), B, Nq, q_pos0, E, m,
        H_I, 2 * half, _ptr(_u16(scores)), _ptr(scores_f32), _stream(dev)))
    return scores, scores_f32


def topk_f32(scores, q_pos0: int, m: int, k: int, topk_idx=None, topk_cnt=None):
    """The selector over FP32 scores [B, Nq, E]. Returns (topk_idx, topk_cnt)."""
    lib = load_library()
    if scores.dtype != torch.float32:
        raise TypeError("FP32 scores are expected")
    B, Nq, E = scores.shape
    dev = scores.device
    if topk_idx is None:
        topk_idx = torch.empty((B, Nq, k), dtype=torch.int32, device=dev)
    if topk_cnt is None:
        topk_cnt = torch.empty((B, Nq), dtype=torch.int32, device=dev)
    _check("csa_topk_f32", lib.csa_topk_f32(_ptr(scores), B, Nq, q_pos0, E, m, k, _ptr(topk_idx),
                                            _ptr(topk_cnt), _stream(dev)))
    return topk_idx, topk_cnt


def topk(scores, q_pos0: int, m: int, k: int, topk_idx=None, topk_cnt=None):
    """Top-k over given BF16 scores [B, Nq, E]."""
    lib = load_library()
    B, Nq, E = scores.shape
    dev = scores.device
    if topk_idx is None:
        topk_idx = torch.empty((B, Nq, k), dtype=torch.int32, device=dev)
    if topk_cnt is None:
        topk_cnt = torch.empty((B, Nq), dtype=torch.int32, device=dev)
    _check("csa_topk", lib.csa_topk(_ptr(_u16(scores)), B, Nq, q_pos0, E, m, k, _ptr(topk_idx),
                                    _ptr(topk_cnt), None, 0, _stream(dev)))
    return topk_idx, topk_cnt


def csa_attend(q, k_cmp, v_cmp, topk_idx, topk_cnt, k_raw, v_raw, W: int, q_pos0: int,
               out=None, lse=None, want_lse: bool = False, ws: Optional[torch.Tensor] = None):
    lib = load_library()
    B, Nq, H, d = q.shape
    E = k_cmp.shape[1]
    N = k_raw.shape[1]
    k = topk_idx.shape[-1]
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty((B, Nq, H), dtype=torch.float32, device=dev)
    need = lib.csa_attend_workspace_size(B, Nq, H, d, k, W)
    ws, wsb = _ws(need, dev, ws)
    _check("csa_attend", lib.csa_attend(
        _ptr(_u16(q)), _ptr(_u16(k_cmp)), _ptr(_u16(v_cmp)), E, _ptr(topk_idx), _ptr(topk_cnt), k,
        _ptr(_u16(k_raw)), _ptr(_u16(v_raw)), N, W, B, Nq, q_pos0, H, d, _ptr(out), _ptr(lse),
        _ptr(ws), wsb, _stream(dev)))
    return out, lse


def hca_attend(q, k_cmp, v_cmp, m: int, k_raw, v_raw, W: int, q_pos0: int, out=None, lse=None,
               want_lse: bool = False, ws: Optional[torch.Tensor] = None):
    lib = load_library()
    B, Nq, H, d = q.shape
    E = k_cmp.shape[1]
    N = k_raw.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty((B, Nq, H), dtype=torch.float32, device=dev)
    need = lib.hca_attend_workspace_size(B, Nq, H, d, E, m, W)
    ws, wsb = _ws(need, dev, ws)
    _check("hca_attend", lib.hca_attend(
        _ptr(_u16(q)), _ptr(_u16(k_cmp)), _ptr(_u16(v_cmp)), E, m, _ptr(_u16(k_raw)),
        _ptr(_u16(v_raw)), N, W, B, Nq, q_pos0, H, d, _ptr(out), _ptr(lse), _ptr(ws), wsb,
        _stream(dev)))
    return out, lse


def _csa_desc(c: Dict) -> CsaLayerDesc:
    q = c["q"]
    B, Nq, H, d = q.shape
    N = c["k_raw"].shape[1]
    H_I, half = c["qi_codes"].shape[2], c["qi_codes"].shape[3]
    dsc = CsaLayerDesc()
    for f in ("q", "k_raw", "v_raw", "logits", "qi_codes", "qi_scales", "ki_codes", "ki_scales",
              "k_cmp", "v_cmp", "out", "lse", "topk_idx", "topk_cnt", "scores", "xi_raw"):
        setattr(dsc, f, _ptr(c.get(f)))
    dsc.B, dsc.Nq, dsc.H, dsc.d = B, Nq, H, d
    dsc.m, dsc.W, dsc.k, dsc.H_I, dsc.d_I = c["m"], c["W"], c["k"], H_I, 2 * half
    dsc.N, dsc.q_pos0, dsc.compress_begin = N, c["q_pos0"], c["compress_begin"]
    return dsc


def _hca_desc(h: Dict) -> HcaLayerDesc:
    q = h["q"]
    B, Nq, H, d = q.shape
    dsc = HcaLayerDesc()
    for f in ("q", "k_raw", "v_raw", "logits", "k_cmp", "v_cmp", "out", "lse"):
        setattr(dsc, f, _ptr(h.get(f)))
    dsc.B, dsc.Nq, dsc.H, dsc.d, dsc.m, dsc.W = B, Nq, H, d, h["m"], h["W"]
    dsc.N, dsc.q_pos0, dsc.compress_begin = h["k_raw"].shape[1], h["q_pos0"], h["compress_begin"]
    return dsc


def layer_pair(csa: Optional[Dict], hca: Optional[Dict], ws: Optional[torch.Tensor] = None):
    """One CSA layer then one HCA layer (either may be None). Dicts hold the tensors named in
    csa_layer_desc / hca_layer_desc plus m, W, k, q_pos0, compress_begin."""
    lib = load_library()
    cd = ctypes.pointer(_csa_desc(csa)) if csa is not None else None
    hd = ctypes.pointer(_hca_desc(hca)) if hca is not None else None
    dev = (csa or hca)["q"].device
    need = lib.csa_hca_layer_pair_workspace_size(cd, hd)
    ws, wsb = _ws(need, dev, ws)
    _check("csa_hca_layer_pair", lib.csa_hca_layer_pair(cd, hd, _ptr(ws), wsb, _stream(dev)))
    return ws


class PreparedLayerPair:
    """A layer-pair call with its descriptors and workspace built once; calling it enqueues one
    csa_hca_layer_pair on torch's current stream. The tensors in `csa` / `hca` stay referenced."""

    def __init__(self, csa: Optional[Dict], hca: Optional[Dict], ws: Optional[torch.Tensor] = None):
        self.lib = load_library()
        self.csa, self.hca = csa, hca
        self.cd = ctypes.pointer(_csa_desc(csa)) if csa is not None else None
        self.hd = ctypes.pointer(_hca_desc(hca)) if hca is not None else None
        self.dev = (csa or hca)["q"].device
        need = self.lib.csa_hca_layer_pair_workspace_size(self.cd, self.hd)
        self.ws, self.wsb = _ws(need, self.dev, ws)
        self.wsp = _ptr(self.ws)

    def __call__(self) -> None:
        _check("csa_hca_layer_pair", self.lib.csa_hca_layer_pair(
            self.cd, self.hd, self.wsp, self.wsb, _stream(self.dev)))


def _paged_desc(L: Dict) -> PagedLayerDesc:
    dsc = PagedLayerDesc()
    dsc.kind = 0 if L["kind"] == "csa" else 1
    B, H, d = L["q"].shape
    dsc.B, dsc.H, dsc.d, dsc.m, dsc.W = B, H, d, L["m"], L["W"]
    dsc.k = L.get("k", 0)
    if dsc.kind == 0:
        dsc.H_I, dsc.d_I = L["qi_codes"].shape[1], 2 * L["qi_codes"].shape[2]
    dsc.N = L["N"]
    for f in ("k_pool", "v_pool", "ki_codes_pool", "ki_scales_pool", "block_table", "ring_k",
              "ring_v", "ring_logits", "ring_xi", "k_new", "v_new", "logit_new", "xi_new", "q",
              "qi_codes", "qi_scales", "out", "lse", "topk_idx", "topk_cnt"):
        setattr(dsc, f, _ptr(L.get(f)))
    dsc.n_pages = L["k_pool"].shape[0]
    dsc.max_blocks = L["block_table"].shape[1]
    return dsc


class PreparedPagedStep:
    """One decode step on a paged cache layer (csa_paged_decode_step): the dict holds the pools,
    rings, block table, the step's token inputs and outputs, and kind ('csa' / 'hca'), m, W, k,
    N (tokens already cached). The descriptor and workspace are built once; calling enqueues the
    step on torch's current stream."""

    def __init__(self, layer: Dict, ws: Optional[torch.Tensor] = None):
        self.lib = load_library()
        self.layer = layer
        self.dsc = ctypes.pointer(_paged_desc(layer))
        self.dev = layer["q"].device
        need = self.lib.csa_paged_decode_workspace_size(self.dsc)
        self.ws, self.wsb = _ws(need, self.dev, ws)
        self.wsp = _ptr(self.ws)

    def __call__(self) -> None:
        _check("csa_paged_decode_step", self.lib.csa_paged_decode_step(
            self.dsc, self.wsp, self.wsb, _stream(self.dev)))


class PreparedPagedPair:
    """One paged decode step of a CSA and an HCA layer (csa_paged_layer_pair: the HCA layer on
    the library's side stream); dicts as for PreparedPagedStep."""

    def __init__(self, csa_layer: Dict, hca_layer: Dict, ws: Optional[torch.Tensor] = None):
        self.lib = load_library()
        self.layers = (csa_layer, hca_layer)
        self.c = ctypes.pointer(_paged_desc(csa_layer))
        self.h = ctypes.pointer(_paged_desc(hca_layer))
        self.dev = csa_layer["q"].device
        need = self.lib.csa_paged_layer_pair_workspace_size(self.c, self.h)
        self.ws, self.wsb = _ws(need, self.dev, ws)
        self.wsp = _ptr(self.ws)

    def __call__(self) -> None:
        _check("csa_paged_layer_pair", self.lib.csa_paged_layer_pair(
            self.c, self.h, self.wsp, self.wsb, _stream(self.dev)))


def paged_decode_step(layer: Dict, ws: Optional[torch.Tensor] = None):
    """One csa_paged_decode_step call on the layer dict (see PreparedPagedStep)."""
    PreparedPagedStep(layer, ws)()


def workspace_sizes(csa: Optional[Dict], hca: Optional[Dict]) -> int:
    lib = load_library()
    cd = ctypes.pointer(_csa_desc(csa)) if csa is not None else None
    hd = ctypes.pointer(_hca_desc(hca)) if hca is not None else None
    return int(lib.csa_hca_layer_pair_workspace_size(cd, hd))


def device_status(reset: bool = True) -> int:
    """Synchronise the current stream and return the device status flags (0 = clean)."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    code = lib.csa_get_device_status(_stream(torch.cuda.current_device()), 1 if reset else 0,
                                     ctypes.byref(flags))
    if code not in (CSA_OK, 7):
        raise CsaError("csa_get_device_status", code)
    return int(flags.value)


def shard_candidates(qi_codes, qi_scales, ki_codes, ki_scales, q_pos0: int, m: int, k: int,
                     ws: Optional[torch.Tensor] = None):
    """One shard's top-k candidates of one query per sequence (csa_shard_candidates): ki_* hold
    the shard's entries [B, E_s, ...]; q_pos0 is the query position relative to the shard's first
    token (t - shard_base * m). Returns (local indices [B, k] int32, BF16 scores [B, k], counts
    [B] int32)."""
    lib = load_library()
    B, Nq, H_I, half = qi_codes.shape
    if Nq != 1:
        raise ValueError("one query per sequence")
    E = ki_codes.shape[1]
    dev = qi_codes.device
    idx = torch.empty((B, k), dtype=torch.int32, device=dev)
    sc = torch.empty((B, k), dtype=torch.bfloat16, device=dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    ws, wsb = _ws(lib.csa_shard_candidates_workspace_size(B, E, k), dev, ws)
    _check("csa_shard_candidates", lib.csa_shard_candidates(
        _ptr(qi_codes), _ptr(qi_scales), _ptr(ki_codes), _ptr(ki_scales), B, q_pos0, E, m, H_I,
        2 * half, k, _ptr(idx), _ptr(_u16(sc)), _ptr(cnt), _ptr(ws), wsb, _stream(dev)))
    return idx, sc, cnt


def topk_merge(cand_scores, cand_idx, cand_cnt, shard_base):
    """The global top-k of S shards' candidates (csa_topk_merge), shard-major: cand_scores
    [S, B, k] bf16, cand_idx [S, B, k] int32 (local), cand_cnt [S, B] int32, shard_base: S
    ascending first global indices (host ints). Returns (topk_idx [B, k] global, topk_cnt [B],
    shard_idx [S, B, k] local, shard_cnt [S, B])."""
    lib = load_library()
    S, B, k = cand_idx.shape
    dev = cand_idx.device
    bases = (ctypes.c_int64 * S)(*[int(x) for x in shard_base])
    idx = torch.empty((B, k), dtype=torch.int32, device=dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    sidx = torch.empty((S, B, k), dtype=torch.int32, device=dev)
    scnt = torch.empty((S, B), dtype=torch.int32, device=dev)
    _check("csa_topk_merge", lib.csa_topk_merge(
        _ptr(_u16(cand_scores)), _ptr(cand_idx), _ptr(cand_cnt), bases, B, S, k, _ptr(idx),
        _ptr(cnt), _ptr(sidx), _ptr(scnt), _stream(dev)))
    return idx, cnt, sidx, scnt


def lse_merge(parts, parts_lse, out=None, lse=None, want_lse: bool = False):
    """Merge S shards' normalised outputs parts [S, ..., d] (bf16) by their log-sum-exp
    parts_lse [S, ...] (csa_lse_merge). Returns (out [..., d] bf16, lse [...] or None)."""
    lib = load_library()
    S = parts.shape[0]
    d = parts.shape[-1]
    rows = parts[0].numel() // d
    dev = parts.device
    if out is None:
        out = torch.empty(parts.shape[1:], dtype=torch.bfloat16, device=dev)
    if want_lse and lse is None:
        lse = torch.empty(parts_lse.shape[1:], dtype=torch.float32, device=dev)
    _check("csa_lse_merge", lib.csa_lse_merge(_ptr(_u16(parts)), _ptr(parts_lse), S, rows, d,
                                              _ptr(out), _ptr(lse), _stream(dev)))
    return out, lse


def _rows_view(t: torch.Tensor):
    """(rows, row_bytes, row_stride_bytes) of a device view whose dimensions after the first
    are contiguous (a whole tensor, or a slice of the second dimension of [B, N, ...])."""
    if not t.is_cuda:
        raise ValueError("tensors must live on the CUDA device")
    es = t.element_size()
    if t.is_contiguous():
        return 1, t.numel() * es, t.numel() * es
    inner = t.shape[1:]
    want, acc = [], 1
    for n in reversed(inner):
        want.append(acc)
        acc *= n
    if t.dim() < 2 or list(t.stride()[1:]) != list(reversed(want)):
        raise ValueError("the view's rows (dimensions after the first) must be contiguous")
    return t.shape[0], acc * es, t.stride(0) * es


def scatter_rows(pairs) -> None:
    """Copy each (dst, src) pair on the device in one launch (csa_scatter_rows): dst a view
    whose dimensions after the first are contiguous (rows strided by its first dimension), src a
    contiguous tensor of the same shape and dtype (rows packed), e.g. slices of one staging
    buffer that a single host-to-device copy filled. At most MAX_COPIES pairs per call."""
    pairs = list(pairs)
    if len(pairs) > MAX_COPIES:
        raise ValueError(f"at most {MAX_COPIES} copies per call")
    descs = (CopyDesc * max(1, len(pairs)))()
    dev = None
    for i, (dst, src) in enumerate(pairs):
        if dst.shape != src.shape or dst.dtype != src.dtype:
            raise ValueError("each source must match its destination's shape and dtype")
        rows, row_bytes, stride = _rows_view(dst)
        descs[i].dst = dst.data_ptr()
        descs[i].src = _ptr(src).value
        descs[i].rows, descs[i].row_bytes, descs[i].dst_stride = rows, row_bytes, stride
        dev = dst.device
    if dev is None:
        return
    _check("csa_scatter_rows", load_library().csa_scatter_rows(descs, len(pairs), _stream(dev)))


FAULT_SKIP_KEY_COPIES = 0x1


def test_set_faults(wait_budget_cycles: int = 0, skip_mask: int = 0) -> None:
    """Failure injection for tests (csa_test_set_faults): a shorter bound on every device-side
    wait and producers that skip their work. (0, 0) restores the defaults."""
    _check("csa_test_set_faults", load_library().csa_test_set_faults(wait_budget_cycles, skip_mask))


def profiler_enable(on: bool = True) -> None:
    """Bracket every kernel launch of the library with CUDA events (tracing aid)."""
    _check("csa_profiler_enable", load_library().csa_profiler_enable(1 if on else 0))


def profiler_collect(reset: bool = True) -> Dict[str, Tuple[int, float]]:
    """{kernel name: (launches, summed device ms)} since the last reset."""
    lib = load_library()
    buf = (KernelTime * 64)()
    n = _I(0)
    _check("csa_profiler_collect", lib.csa_profiler_collect(buf, 64, ctypes.byref(n),
                                                            1 if reset else 0))
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n.value, 64))}
