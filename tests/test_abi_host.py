"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, sizes its workspaces, and rejects bad arguments before
launching anything.  No GPU needed: every call here returns on the host."""

import ctypes
import os
import re

import pytest

from transformer_attention_ggd_gb300 import bam_attn as ba
from transformer_attention_ggd_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bam_attn.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return ba.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bam_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(ba.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert ba.bam_status_string(code) != "unknown status"
    assert ba.bam_status_string(99) == "unknown status"


def test_release_and_debug_builds():
    """The release library reports no debug checks; the BAM_DEBUG build of
    the same sources exports the same symbols and reports its checks.  Both
    queries return on the host."""
    rel = ctypes.CDLL(lib_build.build())
    dbg = ctypes.CDLL(lib_build.build(debug=True))
    assert rel.bam_attn_debug_build() == 0
    assert dbg.bam_attn_debug_build() == 1
    for name in _declared_functions():
        assert hasattr(dbg, name), name


def test_workspace_sizes(lib):
    for op in (ba.BAM_OP_FWD, ba.BAM_OP_BWD, ba.BAM_OP_DECODE):
        n = ba.bam_attn_workspace_size(op, 2, 4, 256, 64)
        assert n > 0 and n % 256 == 0
        assert ba.bam_attn_workspace_size(op, 0, 4, 256, 64) == 0
        assert ba.bam_attn_workspace_size(op, 2, 4, 0, 64) == 0
        assert ba.bam_attn_workspace_size(op, 2, 4, 256, 128) == 0
    assert ba.bam_attn_workspace_size(7, 2, 4, 256, 64) == 0
    # The backward keeps an fp32 dq accumulator: at least B*H*T*64*4 bytes.
    assert ba.bam_attn_workspace_size(ba.BAM_OP_BWD, 8, 12, 512, 64) >= 8 * 12 * 512 * 64 * 4


FAKE = 0x7F0000000000  # 256-aligned, never dereferenced: every call below fails first


def _params(eps=1e-5, causal=1, ssmax=0, s=FAKE, prior=ba.BAM_PRIOR_ALPHA):
    return ba.BamParams(FAKE, FAKE, FAKE, s, eps, causal, ssmax, prior)


def _fwd(lib, q=FAKE, o=FAKE, B=1, H=1, T=16, D=64, p=None, ws=FAKE, ws_bytes=1 << 30):
    p = p or _params()
    vp = ctypes.c_void_p
    return lib.bam_attn_fwd(vp(q), vp(FAKE), vp(FAKE), vp(o), 1, None, B, H, T, D,
                            ctypes.byref(p), vp(ws), ws_bytes, None)


def test_fwd_argument_errors(lib):
    assert _fwd(lib, q=0) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, o=0) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, q=FAKE + 8) == ba.BAM_ERR_INVALID_ARG         # misaligned
    assert _fwd(lib, T=0) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, D=128) == ba.BAM_ERR_UNSUPPORTED
    assert _fwd(lib, p=_params(eps=0.0)) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, p=_params(ssmax=1, s=0)) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, p=_params(causal=2)) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, p=_params(prior=2)) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, p=_params(prior=-1)) == ba.BAM_ERR_INVALID_ARG
    assert _fwd(lib, ws=0) == ba.BAM_ERR_WORKSPACE
    assert _fwd(lib, ws=FAKE + 16) == ba.BAM_ERR_WORKSPACE         # not 256-aligned
    assert _fwd(lib, ws_bytes=100) == ba.BAM_ERR_WORKSPACE
    vp = ctypes.c_void_p
    assert lib.bam_attn_fwd(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, None, 1, 1, 16, 64, None,
                            vp(FAKE), 1 << 30, None) == ba.BAM_ERR_INVALID_ARG


def test_bwd_and_decode_argument_errors(lib):
    vp = ctypes.c_void_p
    p = _params()
    f = [vp(FAKE)] * 3
    # bwd: lse missing
    assert lib.bam_attn_bwd(*f, vp(FAKE), 1, None, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                            vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 1, 16, 64,
                            ctypes.byref(p), vp(FAKE), 1 << 30, None) == ba.BAM_ERR_INVALID_ARG
    # bwd: workspace too small
    assert lib.bam_attn_bwd(*f, vp(FAKE), 1, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                            vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 1, 16, 64,
                            ctypes.byref(p), vp(FAKE), 256, None) == ba.BAM_ERR_WORKSPACE
    # decode: D unsupported, Tkv invalid, workspace small
    assert lib.bam_attn_decode(*f, vp(FAKE), 1, None, 1, 1, 16, 32, ctypes.byref(p), vp(FAKE),
                               1 << 30, None) == ba.BAM_ERR_UNSUPPORTED
    assert lib.bam_attn_decode(*f, vp(FAKE), 1, None, 1, 1, 0, 64, ctypes.byref(p), vp(FAKE),
                               1 << 30, None) == ba.BAM_ERR_INVALID_ARG
    assert lib.bam_attn_decode(*f, vp(FAKE), 1, None, 1, 1, 16, 64, ctypes.byref(p), vp(FAKE),
                               16, None) == ba.BAM_ERR_WORKSPACE


def test_decode_varlen_argument_errors(lib):
    vp = ctypes.c_void_p
    p = _params()
    f = [vp(FAKE)] * 3
    # missing or misaligned cache lengths
    assert lib.bam_attn_decode_varlen(*f, None, vp(FAKE), 1, None, 2, 1, 16, 64, ctypes.byref(p),
                                      vp(FAKE), 1 << 30, None) == ba.BAM_ERR_INVALID_ARG
    assert lib.bam_attn_decode_varlen(*f, vp(FAKE + 2), vp(FAKE), 1, None, 2, 1, 16, 64,
                                      ctypes.byref(p), vp(FAKE), 1 << 30,
                                      None) == ba.BAM_ERR_INVALID_ARG
    # Tmax invalid, workspace too small
    assert lib.bam_attn_decode_varlen(*f, vp(FAKE), vp(FAKE), 1, None, 2, 1, 0, 64,
                                      ctypes.byref(p), vp(FAKE), 1 << 30,
                                      None) == ba.BAM_ERR_INVALID_ARG
    assert lib.bam_attn_decode_varlen(*f, vp(FAKE), vp(FAKE), 1, None, 2, 1, 16, 64,
                                      ctypes.byref(p), vp(FAKE), 16, None) == ba.BAM_ERR_WORKSPACE


def test_decode_paged_argument_errors(lib):
    vp = ctypes.c_void_p
    p = _params()
    f = [vp(FAKE)] * 3

    def call(bt=FAKE, lens=FAKE, page=64, max_blocks=4, num_pages=8, ws_bytes=1 << 30):
        return lib.bam_attn_decode_paged(*f, vp(bt), vp(lens), vp(FAKE), 1, None, 2, 1, page,
                                         max_blocks, num_pages, 64, ctypes.byref(p), vp(FAKE),
                                         ws_bytes, None)
    assert call(bt=0) == ba.BAM_ERR_INVALID_ARG
    assert call(lens=0) == ba.BAM_ERR_INVALID_ARG
    assert call(bt=FAKE + 2) == ba.BAM_ERR_INVALID_ARG
    assert call(page=32) == ba.BAM_ERR_INVALID_ARG
    assert call(page=96) == ba.BAM_ERR_INVALID_ARG
    assert call(max_blocks=0) == ba.BAM_ERR_INVALID_ARG
    assert call(num_pages=0) == ba.BAM_ERR_INVALID_ARG
    assert call(ws_bytes=16) == ba.BAM_ERR_WORKSPACE


def test_selftest_rejects_bad_workspace(lib):
    vp = ctypes.c_void_p
    assert lib.bam_attn_selftest_wait(None, 1 << 20, None) == ba.BAM_ERR_WORKSPACE
    assert lib.bam_attn_selftest_wait(vp(FAKE + 16), 1 << 20, None) == ba.BAM_ERR_WORKSPACE
    assert lib.bam_attn_selftest_wait(vp(FAKE), 128, None) == ba.BAM_ERR_WORKSPACE


def test_profile_events_bounds(lib):
    assert lib.bam_attn_profile_events(-1, None, None) == ba.BAM_ERR_INVALID_ARG
    assert lib.bam_attn_profile_events(ba.BAM_KERNEL_COUNT, None, None) == ba.BAM_ERR_INVALID_ARG
    assert lib.bam_attn_profile_events(ba.BAM_KERNEL_FWD, None, None) == ba.BAM_OK


def test_check_status_rejects_bad_workspace(lib):
    assert lib.bam_attn_check_status(None, None) == ba.BAM_ERR_WORKSPACE
    assert lib.bam_attn_check_status(ctypes.c_void_p(FAKE + 8), None) == ba.BAM_ERR_WORKSPACE


def test_prior_codes_and_params_layout_match_the_header():
    text = open(HEADER).read()
    assert int(re.search(r"BAM_PRIOR_ALPHA\s*=\s*(\d+)", text).group(1)) == ba.BAM_PRIOR_ALPHA
    assert int(re.search(r"BAM_PRIOR_THETA\s*=\s*(\d+)", text).group(1)) == ba.BAM_PRIOR_THETA
    body = re.search(r"typedef struct \{(.*?)\} bam_params;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"(\w+)\s*;", body)
    assert fields == [f[0] for f in ba.BamParams._fields_]
