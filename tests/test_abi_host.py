"""Host-only checks of the C ABI (no GPU): the library loads, exports every
function the header declares, and rejects bad arguments with a status code
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_b300.h")


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_gemms_b300 import build
    build.build()
    import mixture_experts_layer_gemms_b300 as m
    return m


def declared_functions():
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt)))


def test_header_declares_the_calls():
    names = declared_functions()
    for core in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine",
                 "moe_update_bias"):
        assert core in names


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(moe.EXPORTED)


def _shape(moe, **kw):
    base = dict(T=64, d=256, n_routed=16, top_k=4, n_shared=1, d_ff=128,
                dtype=moe.MOE_F32)
    base.update(kw)
    return moe.MoeShape(*[base[k] for k in ("T", "d", "n_routed", "top_k",
                                            "n_shared", "d_ff", "dtype")])


def _ws(moe, shape):
    n = ctypes.c_size_t()
    st = moe.LIB.moe_workspace_size(ctypes.byref(shape), ctypes.byref(n))
    return st, n.value


def test_workspace_size(moe):
    st, n = _ws(moe, _shape(moe))
    assert st == 0 and n > 0 and n % 256 == 0
    # T*K*I elements of H plus histograms, monotone in T
    st2, n2 = _ws(moe, _shape(moe, T=128))
    assert st2 == 0 and n2 > n
    st0, n0 = _ws(moe, _shape(moe, T=0))
    assert st0 == 0


@pytest.mark.parametrize("kw,code", [
    (dict(d=200), 2),                 # d % 128
    (dict(d_ff=100), 2),              # d_ff % 64
    (dict(top_k=17, n_routed=32), 2),
    (dict(top_k=20), 2),              # > n_routed
    (dict(n_shared=9), 2),
    (dict(dtype=1, n_routed=24), 2),  # bf16 needs n_routed % 16 == 0
    (dict(dtype=1, n_routed=512), 2),
    (dict(T=-1), 1),
    (dict(top_k=0), 1),
    (dict(dtype=7), 1),
])
def test_bad_shapes_rejected(moe, kw, code):
    st, _ = _ws(moe, _shape(moe, **kw))
    assert st == code
    assert moe.LIB.moe_status_string(st)
    assert moe.LIB.moe_last_error_detail()


def test_null_and_misaligned_pointers(moe):
    sh = _shape(moe)
    _, n = _ws(moe, sh)
    P = ctypes.c_void_p
    ws = P(4096)          # never dereferenced: validation fails first
    st = moe.LIB.moe_route(ctypes.byref(sh), None, P(256), P(512), P(768),
                           P(1024), P(1280), ws, n, None)
    assert st == 1
    st = moe.LIB.moe_route(ctypes.byref(sh), P(8), P(256), P(512), P(768),
                           P(1024), P(1280), ws, n, None)   # misaligned u
    assert st == 1
    assert b"aligned" in moe.LIB.moe_last_error_detail()


def test_workspace_too_small(moe):
    sh = _shape(moe)
    _, n = _ws(moe, sh)
    P = ctypes.c_void_p
    st = moe.LIB.moe_permute(ctypes.byref(sh), P(256), P(512), P(768),
                             P(1024), P(1280), P(1536), P(1792), P(4096),
                             n - 256, None)
    assert st == 3
    st = moe.LIB.moe_route(ctypes.byref(sh), P(256), P(512), P(768), P(1024),
                           P(1280), P(1536), None, n, None)
    assert st == 3


def test_update_bias_validation(moe):
    P = ctypes.c_void_p
    assert moe.LIB.moe_update_bias(0, P(256), 8, ctypes.c_float(1e-3), P(512),
                                   None) == 1
    assert moe.LIB.moe_update_bias(4, None, 8, ctypes.c_float(1e-3), P(512),
                                   None) == 1
    assert moe.LIB.moe_update_bias(4, P(256), 8, ctypes.c_float(float("nan")),
                                   P(512), None) == 1


def test_combine_bad_dtype(moe):
    sh = _shape(moe)
    P = ctypes.c_void_p
    st = moe.LIB.moe_combine(ctypes.byref(sh), P(256), P(512), P(768),
                             P(1024), P(1280), P(1536), 5, None)
    assert st == 1


def test_status_strings(moe):
    for code in range(7):
        assert moe.LIB.moe_status_string(code)


@pytest.mark.parametrize("G,M,K,code", [
    (0, 1, 4, 1),       # no groups
    (3, 1, 4, 1),       # 16 experts do not split into 3 groups
    (4, 0, 4, 1),       # keep no group
    (4, 5, 4, 1),       # keep more groups than exist
    (128, 1, 1, 1),     # more groups than experts / the 64-group limit
    (4, 1, 5, 1),       # top_k above the 4 experts of one kept group
])
def test_route_grouped_validation(moe, G, M, K, code):
    sh = _shape(moe, top_k=K)
    _, n = _ws(moe, sh)
    P = ctypes.c_void_p
    st = moe.LIB.moe_route_grouped(ctypes.byref(sh), G, M, P(256), P(512),
                                   P(768), P(1024), P(1280), P(1536), P(4096),
                                   n, None)
    assert st == code, moe.LIB.moe_last_error_detail()


def test_fp8_sizes_and_checks(moe):
    sh = _shape(moe, dtype=moe.MOE_FP8, d_ff=256)
    n = ctypes.c_size_t()
    r256 = lambda x: (x + 255) // 256 * 256       # noqa: E731
    # routed gate/up: 2*N*I x d codes, (2NI/128) x (d/128) fp32 scales, and
    # the same scales as UE8M0 bytes with rows padded to 16
    assert moe.LIB.moe_fp8_weight_bytes(ctypes.byref(sh), 0,
                                        ctypes.byref(n)) == 0
    assert n.value == 2 * 16 * 256 * 256 + r256(64 * 2 * 4) + r256(64 * 16)
    assert moe.LIB.moe_fp8_weight_bytes(ctypes.byref(sh), 3,
                                        ctypes.byref(n)) == 0
    assert n.value == 256 * 256 + r256(2 * 2 * 4) + r256(2 * 16)
    assert moe.LIB.moe_fp8_weight_bytes(ctypes.byref(sh), 4,
                                        ctypes.byref(n)) == 1
    assert moe.LIB.moe_x_perm_bytes(ctypes.byref(sh), ctypes.byref(n)) == 0
    A = 64 * 4     # activations: codes, [d/128][A] scales, [A][16] UE8M0
    assert n.value == A * 256 + r256(2 * A * 4) + r256(A * 16)
    bad = _shape(moe, dtype=moe.MOE_FP8, d_ff=192)     # d_ff % 128
    assert _ws(moe, bad)[0] == 2
    P = ctypes.c_void_p
    st = moe.LIB.moe_pack_weights(ctypes.byref(sh), P(256), P(512), P(768),
                                  P(1024), P(1280), P(1536), P(1792),
                                  P(2048), None)
    assert st == 1 and b"moe_pack_weights_fp8" in moe.LIB.moe_last_error_detail()


@pytest.mark.parametrize("dtype_name,part,code,detail", [
    ("MOE_BF16", 3, 1, b"part=3"),
    ("MOE_BF16", -1, 1, b"part=-1"),
    ("MOE_FP8", 1, 2, b"not split"),
    ("MOE_FP8", 2, 2, b"not split"),
])
def test_expert_ffn_part_validation(moe, dtype_name, part, code, detail):
    """A part outside {0, 1, 2}, or a split call of an e4m3 layer, fails
    before anything is launched."""
    sh = _shape(moe, dtype=getattr(moe, dtype_name), d_ff=256)
    _, n = _ws(moe, sh)
    P = ctypes.c_void_p
    st = moe.LIB.moe_expert_ffn_part(ctypes.byref(sh), part, P(256), P(512),
                                     P(768), P(1024), P(1280), P(1536),
                                     P(1792), P(2048), P(2304), P(4096), n,
                                     None)
    assert st == code
    assert detail in moe.LIB.moe_last_error_detail()


# moe_backward's 22 pointer arguments, in order (8, 9: the saved
# pre-activations, which may both be NULL)
ACT, ACT_S = 8, 9


def _bwd_call(moe, sh, ptrs=None, grad=1, ws=None, nbytes=1 << 40):
    P = ctypes.c_void_p
    p = [P(256 * (i + 1)) for i in range(22)] if ptrs is None else ptrs
    return moe.LIB.moe_backward(ctypes.byref(sh), *p, grad,
                                P(1 << 20) if ws is None else ws, nbytes, None)


@pytest.mark.parametrize("over,code,detail", [
    (dict(dtype=0), 2, b"bf16 layers only"),      # fp32 layer
    (dict(dtype=2, d_ff=256), 2, b"bf16 layers only"),   # e4m3 layer
    (dict(dtype=1, d_ff=192), 2, b"multiple of 128"),
])
def test_backward_shape_checks(moe, over, code, detail):
    sh = _shape(moe, **over)
    n = ctypes.c_size_t()
    assert moe.LIB.moe_backward_workspace_size(ctypes.byref(sh),
                                               ctypes.byref(n)) == code
    assert _bwd_call(moe, sh) == code
    assert detail in moe.LIB.moe_last_error_detail()


def test_backward_argument_checks(moe):
    """Every check that needs no GPU: grad dtype, pointers, alignment and
    the workspace, each refused before anything is launched."""
    sh = _shape(moe, dtype=moe.MOE_BF16)
    n = ctypes.c_size_t()
    assert moe.LIB.moe_backward_workspace_size(ctypes.byref(sh),
                                               ctypes.byref(n)) == 0
    # padded rows: at most T*K + 15*N, in 16-row blocks
    A_pad = (64 * 4 + 15 * 16 + 15) // 16 * 16
    assert n.value >= A_pad * 256 * 2 * 4 and n.value % 256 == 0
    P = ctypes.c_void_p
    assert _bwd_call(moe, sh, grad=2) == 1                   # e4m3 grads
    for i in range(22):
        if i == ACT:
            continue               # act NULL: the recomputing path
        ptrs = [P(256 * (k + 1)) for k in range(22)]
        ptrs[i] = None
        assert _bwd_call(moe, sh, ptrs) == 1, i
        assert b"NULL" in moe.LIB.moe_last_error_detail()
    for i in (0, ACT, ACT_S):                                 # misaligned
        ptrs = [P(256 * (k + 1)) for k in range(22)]
        ptrs[i] = P(258)
        assert _bwd_call(moe, sh, ptrs) == 1, i
        assert b"aligned" in moe.LIB.moe_last_error_detail()
    # act and act_shared come together (or not at all)
    ptrs = [P(256 * (k + 1)) for k in range(22)]
    ptrs[ACT] = None
    assert _bwd_call(moe, sh, ptrs) == 1
    assert b"act_shared given without act" in moe.LIB.moe_last_error_detail()
    ptrs[ACT_S] = None                       # neither: only the workspace
    assert _bwd_call(moe, sh, ptrs, nbytes=n.value - 1) == 3
    assert _bwd_call(moe, sh, nbytes=n.value - 1) == 3       # too small
    assert _bwd_call(moe, sh, ws=P(1 << 20 | 8), nbytes=n.value) == 1
    # without shared experts their weights and gradients may be NULL, so
    # the first refusal is the workspace's
    sh0 = _shape(moe, dtype=moe.MOE_BF16, n_shared=0)
    ptrs = [P(256 * (k + 1)) for k in range(22)]
    for i in (ACT_S, 12, 13, 19, 20, 21):
        ptrs[i] = None
    assert _bwd_call(moe, sh0, ptrs, nbytes=0) == 3


def test_expert_ffn_train_validation(moe):
    """The training forward stores pre-activations for bf16 layers only and
    needs act (and act_shared with shared experts); refused before a
    launch."""
    P = ctypes.c_void_p

    def call(sh, act, act_s):
        _, n = _ws(moe, sh)
        p = [P(256 * (k + 1)) for k in range(9)]
        return moe.LIB.moe_expert_ffn_train(ctypes.byref(sh), *p, act, act_s,
                                            P(1 << 20), n, None)

    bf = _shape(moe, dtype=moe.MOE_BF16)
    assert call(bf, None, P(4096)) == 1
    assert b"act is NULL" in moe.LIB.moe_last_error_detail()
    assert call(bf, P(4096), None) == 1
    assert b"act_shared is NULL" in moe.LIB.moe_last_error_detail()
    assert call(bf, P(4100), P(4096)) == 1
    assert b"aligned" in moe.LIB.moe_last_error_detail()
    for dt in (moe.MOE_F32, moe.MOE_FP8):
        assert call(_shape(moe, dtype=dt, d_ff=256), P(4096), P(8192)) == 2
        assert b"bf16 layers only" in moe.LIB.moe_last_error_detail()
