"""CPU-side checks of the C ABI: the libraries build, load without a GPU, export
every function their headers declare, and reject bad arguments on the host
before any CUDA call (so these run here, with no device)."""
import ctypes
import os
import re

import pytest
import torch

import warp_specialized_attention_gb300 as wsa
from warp_specialized_attention_gb300 import build as wsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    wsa_build.build()
    return wsa.load_library()


def _declared(header):
    text = open(os.path.join(INCLUDE, header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)) - {"defined"}


@pytest.mark.parametrize("header,libname", [
    ("wsattn.h", "libwsattn.so"),
    ("wsattn_testing.h", "libwsattn.so"),
    ("wsattn_probes.h", "libwsattn_probes.so"),
])
def test_every_declared_symbol_is_exported(lib, header, libname):
    names = _declared(header)
    assert names, "no declarations parsed from %s" % header
    so = ctypes.CDLL(os.path.join(os.path.dirname(wsa.__file__), libname))
    for n in sorted(names):
        assert hasattr(so, n), "%s declares %s but %s does not export it" % (header, n, libname)


def test_public_header_declares_the_entry_points():
    assert {"fmha_fwd", "fmha_get_device_status", "fmha_status_str",
            "fmha_last_cuda_error", "fmha_version"} <= _declared("wsattn.h")


def test_status_strings(lib):
    for code in range(5):
        assert lib.fmha_status_str(code)
    assert lib.fmha_version() == (0 << 16) | (1 << 8)


# Fake, 16-byte aligned, non-overlapping "device" addresses: validation must
# reject the call before it dereferences or passes them anywhere.
_BASE = 1 << 40


def _ptrs(n_bytes=1 << 30):
    return [_BASE + i * n_bytes for i in range(5)]


def _call(lib, ptrs=None, B=1, H=1, S=128, D=128, causal=0, scale=0.088, dtype=0):
    q, k, v, o, lse = ptrs or _ptrs()
    return lib.fmha_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(B=0), wsa.FMHA_ERR_INVALID_ARG),
    (dict(H=-1), wsa.FMHA_ERR_INVALID_ARG),
    (dict(S=0), wsa.FMHA_ERR_INVALID_ARG),
    (dict(D=0), wsa.FMHA_ERR_INVALID_ARG),
    (dict(D=96), wsa.FMHA_ERR_UNSUPPORTED),
    (dict(D=256), wsa.FMHA_ERR_UNSUPPORTED),
    (dict(dtype=7), wsa.FMHA_ERR_UNSUPPORTED),
    (dict(dtype=wsa.FMHA_E4M3, D=64), wsa.FMHA_ERR_UNSUPPORTED),     # E4M3: D = 128 only
    (dict(dtype=wsa.FMHA_E4M3, S=1000), wsa.FMHA_ERR_UNSUPPORTED),   # transposed V rows: S % 16
    (dict(dtype=wsa.FMHA_E4M3, scale=0.0), wsa.FMHA_ERR_INVALID_ARG),
    (dict(scale=0.0), wsa.FMHA_ERR_INVALID_ARG),
    (dict(scale=-0.1), wsa.FMHA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), wsa.FMHA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), wsa.FMHA_ERR_INVALID_ARG),
    (dict(B=1 << 31), wsa.FMHA_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 16), wsa.FMHA_ERR_INVALID_ARG),
])
def test_bad_sizes_rejected_on_host(lib, kw, expect):
    assert _call(lib, **kw) == expect


def test_null_and_misaligned_pointers_rejected(lib):
    p = _ptrs()
    for i in range(5):
        bad = list(p)
        bad[i] = 0
        assert _call(lib, bad) == wsa.FMHA_ERR_INVALID_ARG
    for i in range(4):  # q, k, v, o need 16-byte alignment
        bad = list(p)
        bad[i] += 8
        assert _call(lib, bad) == wsa.FMHA_ERR_INVALID_ARG
    bad = list(p)
    bad[4] += 2  # lse needs 4-byte alignment
    assert _call(lib, bad) == wsa.FMHA_ERR_INVALID_ARG


def test_overlapping_output_rejected(lib):
    q, k, v, o, lse = _ptrs()
    assert _call(lib, [q, k, v, q + 64, lse]) == wsa.FMHA_ERR_INVALID_ARG
    assert _call(lib, [q, k, v, o, o + 1024]) == wsa.FMHA_ERR_INVALID_ARG


def test_host_entry_validates_before_any_cuda_call(lib):
    host = [_BASE + (10 + i) * (1 << 30) for i in range(5)]
    dev = _ptrs()
    def call(h=host, d=dev, S=128, n_chunks=0):
        return lib.fmha_fwd_host(*h, *d, 1, 2, S, 128, 0, 0.088, 0, n_chunks, None)
    for i in range(5):
        bad = list(host)
        bad[i] = 0
        assert call(h=bad) == wsa.FMHA_ERR_INVALID_ARG
    bad = list(host)
    bad[4] += 1  # host lse must be 4-byte aligned
    assert call(h=bad) == wsa.FMHA_ERR_INVALID_ARG
    bad = list(dev)
    bad[0] += 8  # staging follows fmha_fwd's rules
    assert call(d=bad) == wsa.FMHA_ERR_INVALID_ARG
    assert call(n_chunks=-1) == wsa.FMHA_ERR_INVALID_ARG
    assert call(n_chunks=65) == wsa.FMHA_ERR_INVALID_ARG
    assert call(S=0) == wsa.FMHA_ERR_INVALID_ARG
    overl = list(host)
    overl[3] = overl[0] + 64  # host o overlapping host q
    assert call(h=overl) == wsa.FMHA_ERR_INVALID_ARG


def test_testing_hook_rejects_bad_knobs(lib):
    q, k, v, o, lse = _ptrs()
    args = (q, k, v, o, lse, 1, 1, 128, 128, 0, 0.088, 0, None)
    assert lib.fmha_fwd_testing(*args, 2, 1.0, 8.0) == wsa.FMHA_ERR_INVALID_ARG
    assert lib.fmha_fwd_testing(*args, 0, 0.0, 8.0) == wsa.FMHA_ERR_INVALID_ARG
    assert lib.fmha_fwd_testing(*args, 0, 1000.0, 8.0) == wsa.FMHA_ERR_INVALID_ARG
    assert lib.fmha_fwd_testing(*args, 0, 1.0, -1.0) == wsa.FMHA_ERR_INVALID_ARG
    assert lib.fmha_fwd_testing(*args, 0, 1.0, 16.0) == wsa.FMHA_ERR_INVALID_ARG
    assert lib.fmha_fwd_testing(*args, 0, 1.0, float("nan")) == wsa.FMHA_ERR_INVALID_ARG
    # E4M3 P is stored as 2^(8 - tau) * P: tau above 8 would overflow it
    args8 = (q, k, v, o, lse, 1, 1, 128, 128, 0, 0.088, wsa.FMHA_E4M3, None)
    assert lib.fmha_fwd_testing(*args8, 0, 1.0, 8.5) == wsa.FMHA_ERR_INVALID_ARG


def test_split_hook_rejects_unsupported_splits(lib):
    """Key-split units need full attention, head dim 128 and an even number of
    key blocks; the count is checked against the units before any CUDA call."""
    q, k, v, o, lse = _ptrs()
    def call(S=1024, D=128, causal=0, split=1, B=1, H=2):
        return lib.fmha_fwd_split_testing(q, k, v, o, lse, B, H, S, D, causal, 0.088, 0, None,
                                          split)
    assert call(split=-2) == wsa.FMHA_ERR_INVALID_ARG
    assert call(causal=1) == wsa.FMHA_ERR_UNSUPPORTED
    assert call(D=64) == wsa.FMHA_ERR_UNSUPPORTED
    assert call(S=1152) == wsa.FMHA_ERR_UNSUPPORTED       # 9 key blocks
    assert call(S=128) == wsa.FMHA_ERR_UNSUPPORTED        # 1 key block
    assert call(split=9) == wsa.FMHA_ERR_INVALID_ARG      # 8 units (2 heads x 4)
    assert call(S=0) == wsa.FMHA_ERR_INVALID_ARG
    # 0 and -1 (none, automatic) go on to fmha_fwd's own checks
    assert lib.fmha_fwd_split_testing(0, k, v, o, lse, 1, 2, 1024, 128, 0, 0.088, 0, None,
                                      0) == wsa.FMHA_ERR_INVALID_ARG
    assert lib.fmha_fwd_split_testing(0, k, v, o, lse, 1, 2, 1024, 128, 0, 0.088, 0, None,
                                      -1) == wsa.FMHA_ERR_INVALID_ARG


def test_split_policy(lib):
    """The host's choice of key-split tail units: the remainder of the last
    wave, when it fits in half of the multiprocessors."""
    lib.fmha_fwd_split_policy.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_int]
    lib.fmha_fwd_split_policy.restype = ctypes.c_int64
    pol = lib.fmha_fwd_split_policy
    assert pol(4, 32, 1024, 128, 0, 152) == 56      # 512 units: 3 waves + 56
    assert pol(1, 32, 4096, 128, 0, 152) == 56      # 512 units
    assert pol(4, 32, 16384, 128, 0, 152) == 0      # 8192 units: remainder 136 > 76
    assert pol(2, 16, 2048, 128, 0, 152) == 0       # 256 units: remainder 104 > 76
    assert pol(1, 2, 1024, 128, 0, 152) == 8        # fewer units than SMs: all split
    assert pol(1, 32, 16384, 128, 0, 152) == 72     # 2048 units: remainder 72
    assert pol(4, 32, 1024, 128, 1, 152) == 0       # causal: longest-first order instead
    assert pol(4, 32, 1024, 64, 0, 152) == 0        # head dim 64: one issuer per tile
    assert pol(1, 1, 1152, 128, 0, 152) == 0        # 9 key blocks: odd
    assert pol(1, 1, 128, 128, 0, 152) == 0         # a single key block
    assert pol(4, 32, 1024, 128, 0, 148) == 68      # the count follows the SM count
    assert pol(4, 32, 1024, 128, 0, 0) == -1
    assert pol(0, 32, 1024, 128, 0, 152) == -1


def test_e4m3_overlap_uses_the_byte_sizes(lib):
    """Inputs are 1 byte per element and O 2 bytes: an O that starts inside
    the second half of a same-count 16-bit-sized region of q is still past q's
    E4M3 bytes, so it is accepted up to validation (a CUDA error here, no GPU);
    one that starts inside q's bytes is rejected."""
    q, k, v, o, lse = _ptrs()
    n = 1 * 1 * 128 * 128
    assert _call(lib, [q, k, v, q + n - 16, lse], dtype=wsa.FMHA_E4M3) == wsa.FMHA_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert _call(lib, [q, k, v, q + n, lse], dtype=wsa.FMHA_E4M3) == wsa.FMHA_ERR_CUDA


def test_noalloc_backward_rejects_what_its_scratch_cannot_hold(lib):
    """fmha_bwd_noalloc checks its capacity (96 MiB: B*H*S*(4D + 4) bytes) on
    the host, before any CUDA call."""
    q, k, v, o, lse = _ptrs()
    args = (q, k, v, o, lse, _BASE + 5 * (1 << 30), _BASE + 6 * (1 << 30), _BASE + 7 * (1 << 30),
            _BASE + 8 * (1 << 30))
    cap_rows = (96 << 20) // (4 * 128 + 4)                       # 195,084 at D = 128
    assert lib.fmha_bwd_noalloc(*args, 1, 1, cap_rows + 1, 128, 0, 0.088, 0, None) == \
        wsa.FMHA_ERR_UNSUPPORTED
    assert lib.fmha_bwd_noalloc(*args, 1, 1, 128, 128, 0, 0.088, wsa.FMHA_E4M3, None) == \
        wsa.FMHA_ERR_UNSUPPORTED
    assert lib.fmha_bwd_noalloc(*args, 0, 1, 128, 128, 0, 0.088, 0, None) == \
        wsa.FMHA_ERR_INVALID_ARG
    if not torch.cuda.is_available():   # within capacity: validation passes, CUDA is missing
        assert lib.fmha_bwd_noalloc(*args, 1, 1, cap_rows, 128, 0, 0.088, 0, None) == \
            wsa.FMHA_ERR_CUDA


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    assert _call(lib) == wsa.FMHA_ERR_CUDA
    assert lib.fmha_last_cuda_error()


def test_binding_fails_loudly_without_cuda_tensors(lib):
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        wsa.attention(q, q, q)


def test_no_multicast_or_trap_in_sources():
    """The kernels use no cluster multicast, no trap and no Hopper-only MMA."""
    csrc = os.path.join(ROOT, "warp_specialized_attention_gb300", "csrc")
    banned = ["multicast::cluster", "__trap", "wgmma"]
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        for b in banned:
            assert b not in text, "%s uses %s" % (f, b)


def test_backward_host_entry_validates_before_any_cuda_call(lib):
    host = [_BASE + (10 + i) * (1 << 30) for i in range(9)]   # q k v o lse d_o dq dk dv
    scratch = _BASE + 30 * (1 << 30)
    need = lib.fmha_bwd_host_scratch_bytes(1, 2, 128, 128)

    def call(h=host, sc=scratch, nbytes=need, S=128, n_chunks=0, dtype=0):
        return lib.fmha_bwd_host(*h, sc, nbytes, 1, 2, S, 128, 0, 0.088, dtype, n_chunks, None)
    for i in range(9):
        bad = list(host)
        bad[i] = 0
        assert call(h=bad) == wsa.FMHA_ERR_INVALID_ARG
    bad = list(host)
    bad[4] += 2  # host lse must be 4-byte aligned
    assert call(h=bad) == wsa.FMHA_ERR_INVALID_ARG
    assert call(sc=0) == wsa.FMHA_ERR_INVALID_ARG
    assert call(sc=scratch + 16) == wsa.FMHA_ERR_INVALID_ARG   # scratch: 256-byte aligned
    assert call(nbytes=need - 1) == wsa.FMHA_ERR_INVALID_ARG
    assert call(n_chunks=-1) == wsa.FMHA_ERR_INVALID_ARG
    assert call(n_chunks=65) == wsa.FMHA_ERR_INVALID_ARG
    assert call(S=0) == wsa.FMHA_ERR_INVALID_ARG
    assert call(dtype=wsa.FMHA_E4M3) == wsa.FMHA_ERR_UNSUPPORTED
    overl = list(host)
    overl[6] = overl[0] + 64  # host dq overlapping host q
    assert call(h=overl) == wsa.FMHA_ERR_INVALID_ARG
    if not torch.cuda.is_available():   # valid: the first CUDA call (stream creation) fails
        assert call() == wsa.FMHA_ERR_CUDA


def test_backward_host_scratch_size(lib):
    """Eight (B*H*S*D) 16-bit staging tensors and the (B*H*S) float32 lse, each
    rounded up to 256 bytes, then the workspace of fmha_bwd (B*H*S*(D + 1)
    float32)."""
    def up(x):
        return (x + 255) // 256 * 256
    for B, H, S, D in ((1, 1, 17, 64), (2, 3, 1000, 128), (4, 32, 16384, 128)):
        rows = B * H * S
        want = 8 * up(rows * D * 2) + up(rows * 4) + rows * (D + 1) * 4
        assert lib.fmha_bwd_host_scratch_bytes(B, H, S, D) == want
    assert lib.fmha_bwd_host_scratch_bytes(1, 1, 17, 64) == 23108
    assert lib.fmha_bwd_host_scratch_bytes(0, 1, 128, 64) == 0
