"""GPU checks of the attention kernel's building blocks on one 128-row tile:
the S = Q K^T MMA (K-major SMEM operands from 128-byte-swizzled TMA boxes) and
the O = P V MMA (P from Tensor Memory, V as an MN-major SMEM operand), against
fp64 CPU products of the same 16-bit values."""
import ctypes
import os

import pytest
import torch

import warp_specialized_attention_gb300 as wsa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def probes():
    path = os.path.join(os.path.dirname(wsa.__file__), "libwsattn_probes.so")
    if not os.path.exists(path):
        pytest.fail("libwsattn_probes.so missing: run the build first")
    lib = ctypes.CDLL(path)
    for f in (lib.wsa_probe_qk, lib.wsa_probe_pv):
        f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int]
        f.restype = ctypes.c_int
    for f in (lib.wsa_probe_qk_e4m3, lib.wsa_probe_pv_e4m3):
        f.argtypes = [ctypes.c_void_p] * 3
        f.restype = ctypes.c_int
    for f in (lib.wsa_probe_kmaj_mn, lib.wsa_probe_mn_mn):
        f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int]
        f.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_qk_tile(probes, D, dtype):
    g = torch.Generator().manual_seed(7 + D)
    a = torch.randn(128, D, generator=g).to(dtype)
    b = torch.randn(128, D, generator=g).to(dtype)
    ref = a.double() @ b.double().T
    c = torch.full((128, 128), float("nan"), device="cuda")
    ad, bd = a.cuda(), b.cuda()  # keep both alive: a temporary's memory can be reused
    rc = probes.wsa_probe_qk(ad.data_ptr(), bd.data_ptr(), c.data_ptr(), D,
                             int(dtype == torch.bfloat16))
    assert rc == 0
    err = (c.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "max abs error %g" % err


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_pv_tile(probes, D, dtype):
    g = torch.Generator().manual_seed(11 + D)
    p = torch.rand(128, 128, generator=g).to(dtype)
    v = torch.randn(128, D, generator=g).to(dtype)
    ref = p.double() @ v.double()
    o = torch.full((128, D), float("nan"), device="cuda")
    pd, vd = p.cuda(), v.cuda()
    rc = probes.wsa_probe_pv(pd.data_ptr(), vd.data_ptr(), o.data_ptr(), D,
                             int(dtype == torch.bfloat16))
    assert rc == 0
    err = (o.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "max abs error %g" % err


def _e4m3(x):
    """E4M3 values (torch's float8_e4m3fn: max 448, no infinities) and their bytes."""
    f8 = x.to(torch.float8_e4m3fn)
    return f8.to(torch.float64), f8.view(torch.uint8).contiguous()


def test_qk_tile_e4m3(probes):
    g = torch.Generator().manual_seed(21)
    a, a8 = _e4m3(torch.randn(128, 128, generator=g))
    b, b8 = _e4m3(torch.randn(128, 128, generator=g))
    ref = a @ b.T                      # products of E4M3 values are exact in fp32
    c = torch.full((128, 128), float("nan"), device="cuda")
    ad, bd = a8.cuda(), b8.cuda()
    assert probes.wsa_probe_qk_e4m3(ad.data_ptr(), bd.data_ptr(), c.data_ptr()) == 0
    err = (c.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "max abs error %g" % err


def test_pv_tile_e4m3(probes):
    g = torch.Generator().manual_seed(23)
    p, p8 = _e4m3(torch.rand(128, 128, generator=g) * 4)
    v, v8 = _e4m3(torch.randn(128, 128, generator=g))
    ref = p @ v
    o = torch.full((128, 128), float("nan"), device="cuda")
    pd, vtd = p8.cuda(), v8.T.contiguous().cuda()   # V goes in transposed: vt[d][key]
    assert probes.wsa_probe_pv_e4m3(pd.data_ptr(), vtd.data_ptr(), o.data_ptr()) == 0
    err = (o.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "max abs error %g" % err


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_kmaj_mn_tile(probes, D, dtype):
    """The backward's dK form: A K-major (dS^T), B MN-major (Q)."""
    g = torch.Generator().manual_seed(31 + D)
    a = torch.randn(128, 128, generator=g).to(dtype)
    b = torch.randn(128, D, generator=g).to(dtype)
    ref = a.double() @ b.double()
    c = torch.full((128, D), float("nan"), device="cuda")
    ad, bd = a.cuda(), b.cuda()
    assert probes.wsa_probe_kmaj_mn(ad.data_ptr(), bd.data_ptr(), c.data_ptr(), D,
                                    int(dtype == torch.bfloat16)) == 0
    err = (c.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "max abs error %g" % err


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_mn_mn_tile(probes, D, dtype):
    """The backward's dQ form: A read MN-major from its transpose (the dS^T
    tile read as dS), B MN-major (K)."""
    g = torch.Generator().manual_seed(37 + D)
    a = torch.randn(128, 128, generator=g).to(dtype)
    b = torch.randn(128, D, generator=g).to(dtype)
    ref = a.double() @ b.double()
    c = torch.full((128, D), float("nan"), device="cuda")
    atd, bd = a.T.contiguous().cuda(), b.cuda()
    assert probes.wsa_probe_mn_mn(atd.data_ptr(), bd.data_ptr(), c.data_ptr(), D,
                                  int(dtype == torch.bfloat16)) == 0
    err = (c.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "max abs error %g" % err
