"""Conversions between the oracle's numpy bit patterns and torch device tensors (tests only)."""
import numpy as np
import torch


def to_dev(a, dtype=None):
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    t = torch.from_numpy(a)
    return t.cuda() if dtype is None else t.to(dtype).cuda()


def to_np(t):
    """CUDA tensor -> numpy; bf16 comes back as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def assert_close_bf16(got_u16, want_u16, atol=2e-2, rtol=2e-2, rel_norm=1e-2, what=""):
    """Elementwise |got - want| <= atol + rtol |want| (the bf16 output tolerance), plus a relative
    Frobenius error bound that is meaningful for small-magnitude outputs."""
    g = bf(got_u16).astype(np.float64)
    w = bf(want_u16).astype(np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    bad = np.abs(g - w) > atol + rtol * np.abs(w)
    assert not bad.any(), "%s: %d of %d elements out of tolerance; worst |d|=%g" % (
        what, int(bad.sum()), bad.size, float(np.abs(g - w).max()))
    n = np.linalg.norm(w)
    if n > 0:
        r = np.linalg.norm(g - w) / n
        assert r <= rel_norm, "%s: relative error norm %g > %g" % (what, r, rel_norm)


def assert_same_selection(got, want, what="selection"):
    """Top-k selections, bit for bit as sets: each row of `got` holds exactly the non-negative entries
    of the same row of `want` (the oracle lists them by score), written in ascending position and
    followed by -1 padding (the library's order: the pages leave the order open)."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (got.shape, want.shape)
    for r in range(got.shape[0]):
        g, w = got[r], want[r]
        n = int((w >= 0).sum())
        assert (g[n:] == -1).all() and (g[:n] >= 0).all(), "%s row %d: %d selected, padding %s" % (what, r, n, g[n:][:8])
        assert (np.diff(g[:n]) > 0).all(), "%s row %d: not in ascending position" % (what, r)
        assert np.array_equal(g[:n], np.sort(w[w >= 0])), "%s row %d: the selected sets differ" % (what, r)
