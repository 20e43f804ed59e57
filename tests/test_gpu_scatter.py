"""csa_scatter_rows (the placement of a step's staged inputs into the layer buffers): every
destination byte equals its source byte and nothing else in the destination buffers changes.
Byte work: compared bit for bit with the same placement done by host indexing."""
import numpy as np
import pytest
import torch

import long_context_compressed_pooling_b300 as csa

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _buf(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype.is_floating_point:
        return torch.randn(shape, generator=g).to(dtype)
    return torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(dtype)


@pytest.mark.parametrize("B,N,n_new", [(3, 40, 5), (16, 32768, 1), (2, 1000, 128)])
def test_scatter_rows_places_every_view(B, N, n_new):
    # layer buffers as a decode or prefill step would hold them, and the views it uploads:
    # a whole tensor (queries), rows strided by N (raw K/V rows, logits), packed codes whose
    # row size is not a multiple of 16 bytes (the byte path)
    d, E = 64, N // 4
    host = {
        "q": _buf((B, 1, 8, d), torch.bfloat16, 1),
        "k_raw": _buf((B, N, d), torch.bfloat16, 2),
        "logits": _buf((B, N), torch.float32, 3),
        "codes": _buf((B, E, 7), torch.uint8, 4),
    }
    dev = {k: v.to(DEV) for k, v in host.items()}
    j = max(1, n_new // 4)
    views = [("q", lambda t: t), ("k_raw", lambda t: t[:, N - n_new:]),
             ("logits", lambda t: t[:, N - n_new:]), ("codes", lambda t: t[:, E - j:])]
    new = {name: _buf(tuple(f(host[name]).shape), host[name].dtype, 10 + i)
           for i, (name, f) in enumerate(views)}
    # one packed staging buffer, as one host-to-device copy would fill it
    parts, off = [], 0
    for name, _ in views:
        nb = new[name].numel() * new[name].element_size()
        parts.append((name, off, nb))
        off += (nb + 255) // 256 * 256
    stage = torch.zeros(off, dtype=torch.uint8)
    for name, o, nb in parts:
        stage[o:o + nb] = new[name].contiguous().view(-1).view(torch.uint8)
    dstage = stage.to(DEV)
    pairs = [(f(dev[name]), dstage[o:o + nb].view(new[name].dtype).view(new[name].shape))
             for (name, f), (_, o, nb) in zip(views, parts)]
    csa.scatter_rows(pairs)
    torch.cuda.synchronize()
    for name, f in views:
        f(host[name]).copy_(new[name])  # the expected placement, on the host
        got = dev[name].cpu().contiguous().view(torch.uint8).numpy()
        want = host[name].contiguous().view(torch.uint8).numpy()
        assert np.array_equal(got, want), name
    assert csa.device_status() == 0


def test_scatter_rows_refuses_bad_views():
    t = torch.zeros((4, 8, 16), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError, match="contiguous"):
        csa.scatter_rows([(t[:, :, :8], torch.zeros((4, 8, 8), dtype=torch.bfloat16, device=DEV))])
    with pytest.raises(ValueError, match="shape"):
        csa.scatter_rows([(t, torch.zeros((4, 8, 8), dtype=torch.bfloat16, device=DEV))])
    with pytest.raises(ValueError, match="at most"):
        csa.scatter_rows([(t, t.clone())] * 17)
