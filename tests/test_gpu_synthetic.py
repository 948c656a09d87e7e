"""The device generator of synthetic fp16 normal values (pkv_fill_normal_f16):
deterministic, continuable across calls, standard normal, and equal to a host
restatement of SplitMix64 + Box-Muller up to fp16 rounding."""
import numpy as np
import pytest
import torch

from paged_kv_cache_138_gb300 import ops
from paged_kv_cache_138_gb300._lib import PagedKVError

pytestmark = pytest.mark.gpu


def host_normals(seed, offset, n):
    """SplitMix64 (Steele, Lea and Flood 2014) outputs j // 2 from state seed,
    Box-Muller in float64: cosine for even j, sine for odd j."""
    j = np.arange(offset, offset + n, dtype=np.uint64)
    p = j >> np.uint64(1)
    z = np.uint64(seed) + (p + np.uint64(1)) * np.uint64(0x9e3779b97f4a7c15)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xbf58476d1ce4e5b9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94d049bb133111eb)
    w = z ^ (z >> np.uint64(31))
    u1 = ((w >> np.uint64(40)) + np.uint64(1)).astype(np.float64) / 2.0 ** 24
    u2 = ((w >> np.uint64(16)) & np.uint64(0xFFFFFF)).astype(np.float64) / 2.0 ** 24
    r = np.sqrt(-2.0 * np.log(u1))
    return np.where(j % np.uint64(2) == 0, r * np.cos(2 * np.pi * u2), r * np.sin(2 * np.pi * u2))


def fill(n, seed, offset):
    t = torch.empty(n, dtype=torch.float16, device="cuda")
    ops.fill_normal(t, seed, offset)
    return t


@pytest.mark.parametrize("n,offset", [(1, 0), (7, 3), (8, 0), (4099, 12345), (1 << 20, 1 << 33)])
def test_matches_host_restatement(native_lib, n, offset):
    seed = 0xC0FFEE
    dev = fill(n, seed, offset).cpu().numpy().astype(np.float64)
    host = host_normals(seed, offset, n)
    # fp32 Box-Muller (hardware sine/cosine: ~2^-21 absolute, times r < 5.8,
    # plus the fp32 angle's rounding) rounded to fp16, against float64: one
    # fp16 unit apart plus 1e-5
    tol = np.maximum(np.abs(host), 2.0 ** -14) * 2.0 ** -10 + 1e-5
    assert np.all(np.abs(dev - host) <= tol)


def test_deterministic_and_continuable(native_lib):
    a = fill(100003, 5, 0)
    b = fill(100003, 5, 0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    whole = fill(3 * 4096 + 5, 5, 77)
    parts = torch.empty_like(whole)
    off = 77
    for lo, hi in ((0, 4096), (4096, 8197), (8197, whole.numel())):
        seg = torch.empty(hi - lo, dtype=torch.float16, device="cuda")
        off = ops.fill_normal(seg, 5, off)
        parts[lo:hi] = seg
    assert off == 77 + whole.numel()
    assert torch.equal(whole.view(torch.int16), parts.view(torch.int16))
    assert not torch.equal(fill(4096, 6, 0).view(torch.int16), fill(4096, 5, 0).view(torch.int16))


def test_standard_normal_moments(native_lib):
    x = fill(1 << 22, 11, 0).double()
    n = x.numel()
    assert abs(x.mean().item()) < 5 / n ** 0.5
    assert abs(x.std().item() - 1.0) < 5e-3
    assert torch.isfinite(x).all()
    # tails: Box-Muller with u1 >= 2^-24 bounds |x| by sqrt(2 ln 2^24) ~ 5.77
    assert x.abs().max().item() < 5.8


def test_rejects_misaligned_destination(native_lib):
    t = torch.empty(64, dtype=torch.float16, device="cuda")
    with pytest.raises(PagedKVError):
        ops.fill_normal(t[1:], 1, 0)       # 2-byte offset from an aligned base
