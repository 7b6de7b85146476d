"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/prism.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os

import pytest

from audio_diffusion_dits_zone_b300 import prism as P

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(P.LIB_PATH):
        from audio_diffusion_dits_zone_b300 import build
        build.build()
    return P.lib()


def test_header_declares_the_path(L):
    names = P.header_functions()
    for n in ("prism_zone_shapes", "prism_pool_score", "prism_select", "prism_bsa_fwd", "prism_bsa_bwd",
              "prism_status_check", "prism_last_error", "prism_build_info"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in P.header_functions():
        assert hasattr(L, n), n
    assert set(P.header_functions()) <= set(P._SIGS), "binding misses a declared function"


def test_build_info(L):
    info = P.build_info()
    assert "sm_103a" in info and "tcgen05" in info


def test_library_is_built_for_sm_103a():
    # the object code of every kernel file targets sm_103a (cuobjdump-free check: the
    # build script passes exactly this gencode and nothing else)
    from audio_diffusion_dits_zone_b300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def _sz(n=0):
    return ctypes.byref(ctypes.c_size_t(n))


def test_select_rejects_bad_arguments(L):
    p = ctypes.c_void_p(16)
    assert L.prism_select(p, 1, 0, 0.5, 0.2, p, p, None) == P.PRISM_EINVAL
    assert L.prism_select(p, 1, 5000, 0.5, 0.2, p, p, None) == P.PRISM_EUNSUPPORTED
    assert L.prism_select(p, 1, 10, 1.0, 0.2, p, p, None) == P.PRISM_EINVAL
    assert L.prism_select(p, 1, 10, -0.1, 0.2, p, p, None) == P.PRISM_EINVAL
    assert L.prism_select(p, 1, 10, 0.5, 1.5, p, p, None) == P.PRISM_EINVAL
    assert L.prism_select(None, 1, 10, 0.5, 0.2, p, p, None) == P.PRISM_EINVAL
    assert b"sparsity" in L.prism_last_error() or b"NULL" in L.prism_last_error()


def test_attention_rejects_bad_arguments(L):
    p = ctypes.c_void_p(256)
    # wrong nb
    assert L.prism_bsa_fwd(p, p, p, P.PRISM_BF16, 1024, 1000, 8, 128, 128, p, p, 7, None, p, p, None, _sz(), None) == \
        P.PRISM_EINVAL
    # unsupported head dim / block size
    assert L.prism_bsa_fwd(p, p, p, P.PRISM_BF16, 1024, 1000, 8, 96, 128, p, p, 8, None, p, p, None, _sz(), None) == \
        P.PRISM_EUNSUPPORTED
    assert L.prism_bsa_fwd(p, p, p, P.PRISM_BF16, 1024, 1000, 8, 128, 32, p, p, 32, None, p, p, None, _sz(), None) == \
        P.PRISM_EUNSUPPORTED
    # ld too small
    assert L.prism_bsa_fwd(p, p, p, P.PRISM_BF16, 512, 1000, 8, 128, 128, p, p, 8, None, p, p, None, _sz(), None) == \
        P.PRISM_EINVAL
    # bad dtype
    assert L.prism_bsa_bwd(p, p, p, p, p, p, 7, 1024, 1000, 8, 128, 128, p, p, 8, None, p, p, p, None, _sz(), None) == \
        P.PRISM_EINVAL


def test_workspace_query_needs_no_gpu(L):
    p = ctypes.c_void_p(256)
    n = ctypes.c_size_t(0)
    assert L.prism_bsa_fwd(p, p, p, P.PRISM_BF16, 1024, 1000, 8, 128, 128, p, p, 8, None, p, p, None, ctypes.byref(n),
                           None) == P.PRISM_OK
    assert n.value >= 256 and n.value % 256 == 0
    m = ctypes.c_size_t(0)
    assert L.prism_bsa_bwd(p, p, p, p, p, p, P.PRISM_BF16, 1024, 1000, 8, 128, 128, p, p, 8, None, p, p, p, None,
                           ctypes.byref(m), None) == P.PRISM_OK
    # transposed lists (bits + counts + indices) and the row term D
    assert m.value >= 8 * 8 * 8 * 4 + 8 * 1000 * 4
    shapes = (ctypes.c_int32 * 12)(1, 8, 16, 2, 8, 8, 4, 4, 8, 8, 4, 4)
    z = ctypes.c_size_t(0)
    assert L.prism_zone_shapes(p, P.PRISM_BF16, 5120, 5120, p, 21, 45, 80, 3, 9, 16, shapes, 4, p, p, None,
                               ctypes.byref(z), None) == P.PRISM_OK
    assert z.value >= 175 * 3 * 4
    # zones too large to stage
    assert L.prism_zone_shapes(p, P.PRISM_BF16, 64, 64, p, 64, 64, 64, 64, 64, 64, shapes, 4, p, p, None,
                               ctypes.byref(z), None) == P.PRISM_EUNSUPPORTED


def test_pool_score_argument_rules(L):
    p = ctypes.c_void_p(256)
    # copies without perm
    assert L.prism_pool_score(p, p, p, P.PRISM_BF16, 1024, None, 1000, 8, 128, 128, p, None, None, 1024, p, p, p,
                              None) == P.PRISM_EINVAL
    # scores without block means
    assert L.prism_pool_score(p, p, p, P.PRISM_BF16, 1024, None, 1000, 8, 128, 128, None, None, None, 0, None, None,
                              p, None) == P.PRISM_EINVAL


def test_a2v_norm_argument_rules_and_workspace(L):
    p = ctypes.c_void_p(256)
    n = ctypes.c_size_t(0)
    # workspace: one fp32 squared norm per (head, video token)
    assert L.prism_a2v_norm(p, p, p, P.PRISM_BF16, 5120, 5120, 75600, 157, 40, 128, None, p, None, ctypes.byref(n),
                            None) == P.PRISM_OK
    assert n.value >= 40 * 75600 * 4 and n.value % 256 == 0
    # only bf16 with d = 128 is built
    assert L.prism_a2v_norm(p, p, p, P.PRISM_F32, 5120, 5120, 75600, 157, 40, 128, None, p, None, _sz(),
                            None) == P.PRISM_EUNSUPPORTED
    assert L.prism_a2v_norm(p, p, p, P.PRISM_BF16, 2560, 2560, 75600, 157, 40, 64, None, p, None, _sz(),
                            None) == P.PRISM_EUNSUPPORTED
    # sizes, strides, pointers
    assert L.prism_a2v_norm(p, p, p, P.PRISM_BF16, 5120, 5120, 75600, 0, 40, 128, None, p, None, _sz(),
                            None) == P.PRISM_EINVAL
    assert L.prism_a2v_norm(p, p, p, P.PRISM_BF16, 4096, 5120, 75600, 157, 40, 128, None, p, None, _sz(),
                            None) == P.PRISM_EINVAL
    assert L.prism_a2v_norm(p, p, p, P.PRISM_BF16, 5124, 5120, 75600, 157, 40, 128, None, p, None, _sz(),
                            None) == P.PRISM_EINVAL
    ws = ctypes.c_void_p(1 << 20)
    big = ctypes.c_size_t(1 << 30)
    assert L.prism_a2v_norm(None, p, p, P.PRISM_BF16, 5120, 5120, 75600, 157, 40, 128, None, p, ws,
                            ctypes.byref(big), None) == P.PRISM_EINVAL
    assert L.prism_a2v_norm(ctypes.c_void_p(258), p, p, P.PRISM_BF16, 5120, 5120, 75600, 157, 40, 128, None, p, ws,
                            ctypes.byref(big), None) == P.PRISM_EINVAL
    assert b"aligned" in L.prism_last_error()


def test_zone_chunked_sizes_closed_form(L):
    # host only: 720p: 175 zones of 432 tokens, 4 blocks each; 1080p: 7 planes of
    # 49 x 4 + 7 x 2 + 7 x 2 + 1 blocks (zones clipped to 5 rows / 8 columns at the edges)
    nb, np_ = ctypes.c_int32(0), ctypes.c_int64(0)
    assert L.prism_zone_chunked_size(21, 45, 80, 3, 9, 16, 128, ctypes.byref(nb), ctypes.byref(np_)) == P.PRISM_OK
    assert (nb.value, np_.value) == (700, 700 * 128)
    assert L.prism_zone_chunked_size(21, 68, 120, 3, 9, 16, 128, ctypes.byref(nb), ctypes.byref(np_)) == P.PRISM_OK
    assert (nb.value, np_.value) == (7 * 225, 7 * 225 * 128)
    assert L.prism_zone_chunked_size(21, 68, 120, 3, 9, 16, 0, ctypes.byref(nb), ctypes.byref(np_)) == P.PRISM_EINVAL
    shapes = (ctypes.c_int32 * 12)(1, 8, 16, 2, 8, 8, 4, 4, 8, 8, 4, 4)
    z = ctypes.c_size_t(0)
    assert L.prism_zone_perm_chunked(None, 21, 45, 80, 3, 9, 16, shapes, 4, 128, None, None, None, ctypes.byref(z),
                                     None) == P.PRISM_OK
    assert z.value >= 175 * 4
    # the padded block order is whole blocks
    p = ctypes.c_void_p(256)
    assert L.prism_pool_score_chunked(p, p, p, P.PRISM_BF16, 1024, 1000, p, 1100, 8, 128, 128, None, None, None, 0,
                                      p, p, None, None) == P.PRISM_EINVAL
