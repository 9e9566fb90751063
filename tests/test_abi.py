"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports every
entry point declared in include/*.h, and rejects bad arguments on the host
with a message naming the argument (no GPU needed: validation runs before any
device access)."""
import ctypes
import glob
import os
import re

import pytest

import sliding_window_attention_sdpa_gb300 as swa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    swa._build.build()
    return swa.load()


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(sdpa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "sdpa_bwd" in names and "sdpa_bwd_preprocess" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(swa.ENTRY_POINTS)


def test_params_struct_matches_binding(lib):
    assert lib.sdpa_bwd_params_bytes() == ctypes.sizeof(swa.SdpaBwdParams)
    assert lib.sdpa_bwd_tile_kv() == 128 and lib.sdpa_bwd_tile_q() == 128


def base_params(**kw):
    p = swa.SdpaBwdParams()
    p.dtype, p.layout, p.mask_mode = swa.SDPA_BF16, swa.SDPA_BSHD, swa.SDPA_MASK_TOP_LEFT
    p.b, p.h_q, p.h_kv, p.s_q, p.s_kv, p.d = 2, 4, 4, 256, 256, 64
    p.window_left, p.window_right, p.scale = 32, -1, 0.125
    st = swa._i64x3(256 * 4 * 64, 4 * 64, 64)
    for f in ("q", "k", "v", "o", "dout", "dq", "dk", "dv"):
        setattr(p, f + "_stride" if f != "dout" else "do_stride", st)
        setattr(p, f, 4096)
    p.lse = 4096
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_deterministic_slots_workspace():
    """Deterministic mode 1 adds one fp32 128 x d tile per (sequence, q-head,
    q-tile, possible visitor) when a q-tile can have three or more visitors;
    mode 2 (relay only) and two-visitor windows add nothing."""
    wide = dict(window_left=-1, s_q=512, s_kv=512)
    base = swa.sdpa_bwd_workspace_bytes(base_params(**wide))
    relay = swa.sdpa_bwd_workspace_bytes(base_params(deterministic=2, **wide))
    slots = swa.sdpa_bwd_workspace_bytes(base_params(deterministic=1, **wide))
    assert relay == base
    p = base_params(**wide)
    # 4 kv-tiles may visit each of the 4 q-tiles
    extra = p.b * p.h_q * 4 * 4 * 128 * p.d * 4
    assert base + extra <= slots <= base + extra + 256
    # W = 200 over 4 kv-tiles: a q-tile's rows reach back 200 keys, so up to
    # 1 + ceil(200 / 128) = 3 kv-tiles visit it
    s512 = dict(s_q=512, s_kv=512, window_left=200)
    assert (swa.sdpa_bwd_workspace_bytes(base_params(deterministic=1, **s512))
            > swa.sdpa_bwd_workspace_bytes(base_params(**s512)))
    # W = 32: at most 1 + ceil(32 / 128) = 2 visitors (the strip-mode kernel
    # combines them without slots), at either length
    for extra_kw in (dict(s_q=512, s_kv=512), {}):
        assert (swa.sdpa_bwd_workspace_bytes(base_params(deterministic=1, **extra_kw))
                == swa.sdpa_bwd_workspace_bytes(base_params(**extra_kw)))


def test_workspace_bytes():
    p = base_params()
    n = swa.sdpa_bwd_workspace_bytes(p)
    # dQ accumulator alone is b*s*h*d*4 bytes
    assert n >= 2 * 256 * 4 * 64 * 4
    # GQA needs no group-sum buffer (the sum is formed in tensor memory); the
    # one part that follows the kv-heads is the main kernel's item table,
    # 152 bytes per (sequence, kv-head, kv-tile)
    g = base_params(h_kv=2)
    n_kv_tiles = (p.s_kv + 127) // 128
    table_diff = p.b * (p.h_kv - 2) * n_kv_tiles * 152
    assert abs((n - swa.sdpa_bwd_workspace_bytes(g)) - table_diff) < 256
    # d = 128 decodes its items in place: no table, so GQA changes nothing
    n128 = swa.sdpa_bwd_workspace_bytes(base_params(d=128))
    assert n128 > 0 and swa.sdpa_bwd_workspace_bytes(base_params(d=128, h_kv=2)) == n128
    assert swa.sdpa_bwd_workspace_bytes(base_params(d=96)) == 0
    assert "d=96" in swa.last_error()


@pytest.mark.parametrize("field,value,code,needle", [
    ("dtype", 7, swa.SDPA_ERR_INVALID_ARG, "dtype"),
    ("layout", 3, swa.SDPA_ERR_INVALID_ARG, "layout"),
    ("mask_mode", 9, swa.SDPA_ERR_INVALID_ARG, "mask_mode"),
    ("h_kv", 3, swa.SDPA_ERR_INVALID_ARG, "multiple of h_kv"),
    ("d", 80, swa.SDPA_ERR_UNSUPPORTED, "d=80"),
    ("window_left", -5, swa.SDPA_ERR_INVALID_ARG, "window_left"),
    ("deterministic", 3, swa.SDPA_ERR_INVALID_ARG, "deterministic"),
    ("sink", 4096, swa.SDPA_ERR_INVALID_ARG, "dsink"),
    ("scale", 0.0, swa.SDPA_ERR_INVALID_ARG, "scale"),
])
def test_host_validation(field, value, code, needle):
    p = base_params(**{field: value})
    for fn in (swa.sdpa_bwd_preprocess, swa.sdpa_bwd, swa.sdpa_bwd_dq_convert,
               swa.sdpa_bwd_gqa_reduce):
        assert fn(p, 0, 0, None) == code
        assert needle in swa.last_error()


def test_bad_stride_and_workspace():
    p = base_params()
    p.k_stride = swa._i64x3(256 * 4 * 64, 4 * 64 + 3, 64)
    assert swa.sdpa_bwd(p, 0, 0, None) == swa.SDPA_ERR_INVALID_ARG
    assert "k_stride[1]" in swa.last_error()
    p = base_params()
    assert swa.sdpa_bwd(p, 0, 0, None) == swa.SDPA_ERR_WORKSPACE
    assert swa.sdpa_bwd(p, 256, 16, None) == swa.SDPA_ERR_WORKSPACE
    assert "need" in swa.last_error()


def test_bottom_right_with_longer_queries_is_accepted():
    # the first s_q - s_kv rows reach no key; the shape passes validation and
    # only the (missing) workspace is refused
    p = base_params(mask_mode=swa.SDPA_MASK_BOTTOM_RIGHT, s_q=512)
    assert swa.sdpa_bwd(p, 0, 0, None) == swa.SDPA_ERR_WORKSPACE


def test_thd_needs_offsets():
    p = base_params(layout=swa.SDPA_THD, total_q=300, total_kv=300)
    assert swa.sdpa_bwd(p, 0, 0, None) == swa.SDPA_ERR_INVALID_ARG
    assert "offsets" in swa.last_error()


def test_kernel_launch_count():
    """The four calls launch the preprocess, the main kernel and, when some dQ
    row is not written by the main kernel (or dSink needs finishing), the
    convert kernel; gqa_reduce launches nothing."""
    # top-left causal W=32 over 256 rows: every q-tile has one or two visitors
    assert swa.sdpa_bwd_kernel_launches(base_params()) == 2
    # GQA changes nothing
    assert swa.sdpa_bwd_kernel_launches(base_params(h_kv=2)) == 2
    # dSink is finished by the convert kernel
    assert swa.sdpa_bwd_kernel_launches(base_params(sink=4096, dsink=4096)) == 3
    # with length arrays rows past a sequence's length may need zeros
    assert swa.sdpa_bwd_kernel_launches(base_params(seq_q_lens=4096)) == 3
    # no window over 512 rows: q-tile 3 has four visitors, added with atomics
    # (converted by the convert kernel); deterministic mode 1 keeps a partial
    # per visitor, summed by the convert kernel; mode 2 passes the tile along
    # the relay, whose last turn converts
    wide = dict(window_left=-1, s_q=512, s_kv=512)
    assert swa.sdpa_bwd_kernel_launches(base_params(**wide)) == 3
    assert swa.sdpa_bwd_kernel_launches(base_params(deterministic=1, **wide)) == 3
    assert swa.sdpa_bwd_kernel_launches(base_params(deterministic=2, **wide)) == 2
    # bottom-right, 128 queries against 512 keys, W=32: q-tile 0 is visited by
    # kv-tiles 2 and 3 only
    br = dict(mask_mode=swa.SDPA_MASK_BOTTOM_RIGHT, s_q=128, s_kv=512)
    assert swa.sdpa_bwd_kernel_launches(base_params(**br)) == 2
    # no query rows: only the main kernel runs (it writes dK = dV = 0)
    assert swa.sdpa_bwd_kernel_launches(base_params(s_q=0)) == 1
    assert swa.sdpa_bwd_kernel_launches(base_params(d=96)) == -1


def test_forward_params_struct_matches_binding(lib):
    assert lib.sdpa_fwd_params_bytes() == ctypes.sizeof(swa.SdpaFwdParams)


def fwd_params(**kw):
    p = swa.SdpaFwdParams()
    p.dtype, p.layout, p.mask_mode = swa.SDPA_BF16, swa.SDPA_BSHD, swa.SDPA_MASK_TOP_LEFT
    p.b, p.h_q, p.h_kv, p.s_q, p.s_kv, p.d = 2, 4, 4, 256, 256, 64
    p.window_left, p.window_right, p.scale = 32, -1, 0.125
    st = swa._i64x3(256 * 4 * 64, 4 * 64, 64)
    for f in ("q", "k", "v", "o"):
        setattr(p, f + "_stride", st)
        setattr(p, f, 4096)
    p.lse = 4096
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value,code,needle", [
    ("dtype", 7, swa.SDPA_ERR_INVALID_ARG, "dtype"),
    ("layout", 3, swa.SDPA_ERR_INVALID_ARG, "layout"),
    ("mask_mode", 9, swa.SDPA_ERR_INVALID_ARG, "mask_mode"),
    ("h_kv", 3, swa.SDPA_ERR_INVALID_ARG, "multiple of h_kv"),
    ("d", 80, swa.SDPA_ERR_UNSUPPORTED, "d=80"),
    ("window_right", -7, swa.SDPA_ERR_INVALID_ARG, "window_right"),
    ("scale", 0.0, swa.SDPA_ERR_INVALID_ARG, "scale"),
])
def test_forward_host_validation(field, value, code, needle):
    assert swa.sdpa_fwd(fwd_params(**{field: value}), None) == code
    assert needle in swa.last_error()


def test_forward_bad_stride_and_thd_offsets():
    p = fwd_params()
    p.o_stride = swa._i64x3(256 * 4 * 64, 4 * 64 + 3, 64)
    assert swa.sdpa_fwd(p, None) == swa.SDPA_ERR_INVALID_ARG
    assert "o_stride[1]" in swa.last_error()
    p = fwd_params(layout=swa.SDPA_THD, total_q=300, total_kv=300)
    assert swa.sdpa_fwd(p, None) == swa.SDPA_ERR_INVALID_ARG
    assert "offsets" in swa.last_error()
