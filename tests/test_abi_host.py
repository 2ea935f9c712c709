"""The C-ABI library on the host, without a GPU.

Checks that libconvbnsilu.so builds, loads and exports every function that
include/*.h declares, and exercises the entry points that touch no GPU:
output sizes, the tile planner, and argument validation (every invalid call
must return its status code before any CUDA call is made).
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from conv2d_batchnorm_silu_gb300 import _build
    _build.build()
    from conv2d_batchnorm_silu_gb300 import capi
    return capi


def declared_functions():
    names = []
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            if m.group(1) not in ("if", "return", "sizeof"):
                names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("conv_bn_silu_fold", "conv_bn_silu_forward", "conv_bn_silu_output_dims"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_output_dims(lib):
    assert lib.output_dims(640, 640, 3, 3, 2, 1) == (320, 320)
    assert lib.output_dims(160, 160, 3, 3, 2, 1) == (80, 80)
    assert lib.output_dims(40, 40, 1, 1, 1, 0) == (40, 40)
    assert lib.output_dims(20, 20, 3, 3, 1, 1) == (20, 20)
    assert lib.output_dims(7, 9, 3, 2, (2, 3), (0, 1)) == (3, 4)
    assert lib.output_dims(1, 1, 3, 3, 1, 1) == (1, 1)
    for bad in [(0, 5, 1, 1, 1, 0), (5, 5, 3, 3, 0, 0), (5, 5, 3, 3, 1, -1), (2, 2, 3, 3, 1, 0)]:
        with pytest.raises(lib.CbsError):
            lib.output_dims(*bad)


def test_plan_for_the_five_layers(lib):
    from conv2d_batchnorm_silu_gb300.synthetic import LAYERS
    expect_algo = {"tiny": "tcgen05", "stem": "tcgen05", "down": "tcgen05",
                   "pointwise": "tcgen05", "deep": "tcgen05"}
    for name, sh in LAYERS.items():
        p = lib.plan(sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad, "auto", 152)
        assert p["algo"] == expect_algo[name], (name, p)
        if name == "stem":
            # thin-input tensor-core kernel: K = 27 zero-padded to 32, three CTAs per SM
            assert p["block_m"] == 128 and p["block_n"] == 16 and p["block_k"] == 32
            assert p["tiles"] == 800 and p["grid"] == 456 and 3 * (p["smem_bytes"] + 1024) <= 228 * 1024
            continue
        if name in ("down", "pointwise"):
            # channel-major tiles, x in boxes of whole output rows (the 1x1 layer: of its
            # [M][C] matrix), weights loaded with every K step; units of block_m pixels
            assert p["swap_ab"] == 1 and p["row_boxes"] == 1 and p["weights_resident"] == 0, p
            assert p["block_m"] % 16 == 0 and p["block_m"] <= 256 and p["block_n"] == 128
            assert p["grid"] == 152 and p["stream_k"] == 0 and p["cluster"] == 1
            assert p["smem_bytes"] <= 232448 and p["stages"] >= 3
            continue
        if p["algo"] == "tcgen05":
            assert p["swap_ab"] == 0
            assert p["block_m"] == 128
            assert p["block_n"] % 16 == 0 and p["block_n"] <= 256
            assert p["block_n"] >= min(sh.k, 128)
            assert p["stream_k"] == (1 if name == "deep" else 0)
            if p["stream_k"]:
                assert p["block_n"] == 256 and p["grid"] == 152
                assert p["cluster"] == 2
                assert p["workspace_bytes"] >= 150 * 128 * 256 * 4
                # 2-CTA pair tiles: twelve epilogue warps (three per TMEM lane quarter)
                assert p["threads"] == 512 and p["stages"] == 5
            else:
                assert p["threads"] == (384 if p["block_n"] >= 64 else 256)
            assert p["grid"] <= 152 and (p["balanced"] or p["grid"] <= p["tiles"])
            assert p["smem_bytes"] <= 232448
            assert p["stages"] >= 2
            assert p["k_iters"] == sh.r * sh.s * -(-sh.c // p["block_k"])
            tiles = -(-sh.m // p["block_m"]) * -(-sh.k // p["block_n"])
            assert p["tiles"] == tiles


def test_plan_rejects_what_tcgen05_cannot_run(lib):
    with pytest.raises(lib.CbsError) as e:
        lib.plan(1, 64, 64, 5, 16, 3, 3, 2, 1, "tcgen05", 152)   # c = 5: neither TMA nor gather
    assert e.value.status == lib.CBS_ERR_UNSUPPORTED
    # a 3-channel stem is taken by the thin-input tensor-core kernel
    assert lib.plan(1, 64, 64, 3, 16, 3, 3, 2, 1, "tcgen05", 152)["algo"] == "tcgen05"
    with pytest.raises(lib.CbsError):
        lib.plan(1, 64, 64, 16, 12, 3, 3, 1, 1, "tcgen05", 152)  # c_out % 8 != 0
    assert lib.plan(1, 64, 64, 3, 16, 3, 3, 2, 1, "direct", 152)["algo"] == "direct"
    # the thin-input kernel takes a padding of at most 2 (every output row then reads an
    # input row); a larger one goes to the direct kernel
    assert lib.plan(1, 64, 64, 3, 16, 3, 3, 1, 2, "tcgen05", 152)["algo"] == "tcgen05"
    with pytest.raises(lib.CbsError):
        lib.plan(1, 64, 64, 3, 16, 3, 3, 1, 3, "tcgen05", 152)
    assert lib.plan(1, 64, 64, 3, 16, 3, 3, 1, 3, "auto", 152)["algo"] == "direct"


def test_invalid_arguments_return_status_without_gpu(lib):
    f = lib.raw_status
    P = ctypes.c_void_p
    good = P(0x10000)
    odd = P(0x10008)
    # null pointer
    assert f("conv_bn_silu_forward", None, good, good, good, good, 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1,
             None) == lib.CBS_ERR_INVALID_ARG
    # misaligned pointer
    assert f("conv_bn_silu_forward", good, odd, good, good, good, 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1,
             None) == lib.CBS_ERR_MISALIGNED
    # bad dims / stride / pad / kernel larger than padded input
    for dims in [(1, 0, 8, 16, 16, 3, 3, 1, 1, 1, 1), (1, 8, 8, 0, 16, 3, 3, 1, 1, 1, 1),
                 (1, 8, 8, 16, 16, 3, 3, 0, 1, 1, 1), (1, 8, 8, 16, 16, 3, 3, 1, 1, -1, 1),
                 (1, 2, 2, 16, 16, 5, 5, 1, 1, 0, 0), (-1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1)]:
        assert f("conv_bn_silu_forward", good, good, good, good, good, *dims, None) == \
            lib.CBS_ERR_INVALID_ARG
    # bad algorithm id
    assert f("conv_bn_silu_forward_algo", good, good, good, good, good, 1, 8, 8, 16, 16, 3, 3, 1, 1,
             1, 1, 7, None) == lib.CBS_ERR_INVALID_ARG
    # unsupported shape for a forced tcgen05 call, rejected before any launch
    assert f("conv_bn_silu_forward_algo", good, good, good, good, good, 1, 8, 8, 5, 16, 3, 3, 1, 1,
             1, 1, 1, None) == lib.CBS_ERR_UNSUPPORTED
    # empty batch / no output channels are no-ops even with null pointers
    assert f("conv_bn_silu_forward", None, None, None, None, None, 0, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1,
             None) == lib.CBS_OK
    assert f("conv_bn_silu_forward", None, None, None, None, None, 2, 8, 8, 16, 0, 3, 3, 1, 1, 1, 1,
             None) == lib.CBS_OK
    # allocation-free forward: validated like conv_bn_silu_forward, before any CUDA call
    na = "conv_bn_silu_forward_noalloc"
    for nulls in [(None, good, good, good, good), (good, None, good, good, good),
                  (good, good, None, good, good), (good, good, good, None, good),
                  (good, good, good, good, None)]:
        assert f(na, *nulls, 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, None) == lib.CBS_ERR_INVALID_ARG
    for odds in [(odd, good, good, good, good), (good, good, good, good, odd)]:
        assert f(na, *odds, 1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, None) == lib.CBS_ERR_MISALIGNED
    assert f(na, good, good, good, good, good, 1, 8, 8, 16, 16, 3, 3, 0, 1, 1, 1, None) == \
        lib.CBS_ERR_INVALID_ARG
    assert f(na, None, None, None, None, None, 0, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, None) == lib.CBS_OK
    assert f(na, None, None, None, None, None, 2, 8, 8, 16, 0, 3, 3, 1, 1, 1, 1, None) == lib.CBS_OK
    # unfused comparator: t1/t2 are checked like y
    uf = "conv_bn_silu_forward_unfused"
    dims = (1, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1)
    assert f(uf, good, good, good, good, None, good, good, *dims, None) == lib.CBS_ERR_INVALID_ARG
    assert f(uf, good, good, good, good, good, odd, good, *dims, None) == lib.CBS_ERR_MISALIGNED
    assert f(uf, None, None, None, None, None, None, None, 0, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1,
             None) == lib.CBS_OK
    bn_apply = lib._lib.conv_bn_silu_bn_apply
    assert bn_apply(good, good, good, good, 100, 16, None) == lib.CBS_ERR_INVALID_ARG   # 100 % 16
    assert bn_apply(good, good, good, good, 64, 0, None) == lib.CBS_ERR_INVALID_ARG
    assert bn_apply(good, odd, good, good, 64, 16, None) == lib.CBS_ERR_MISALIGNED
    assert bn_apply(None, None, None, None, 0, 16, None) == lib.CBS_OK
    silu_apply = lib._lib.conv_bn_silu_silu_apply
    assert silu_apply(good, good, -1, None) == lib.CBS_ERR_INVALID_ARG
    assert silu_apply(good, None, 8, None) == lib.CBS_ERR_INVALID_ARG
    assert silu_apply(odd, good, 8, None) == lib.CBS_ERR_MISALIGNED
    assert silu_apply(None, None, 0, None) == lib.CBS_OK
    # other epilogues: bad activation id, misaligned residual
    act = "conv_bn_act_forward"
    assert f(act, good, good, good, good, None, good, *dims, 7, None) == lib.CBS_ERR_INVALID_ARG
    assert f(act, good, good, good, good, None, good, *dims, -1, None) == lib.CBS_ERR_INVALID_ARG
    assert f(act, good, good, good, good, odd, good, *dims, 2, None) == lib.CBS_ERR_MISALIGNED
    assert f(act, good, good, good, good, good, None, *dims, 1, None) == lib.CBS_ERR_INVALID_ARG
    assert f(act, None, None, None, None, None, None, 0, 8, 8, 16, 16, 3, 3, 1, 1, 1, 1, 0,
             None) == lib.CBS_OK
    # fp8 output: bad activation id, misaligned output
    f8 = "conv_bn_act_forward_fp8"
    assert f(f8, good, good, good, good, good, *dims, 3, None) == lib.CBS_ERR_INVALID_ARG
    assert f(f8, good, good, good, good, odd, *dims, 0, None) == lib.CBS_ERR_MISALIGNED
    # batched fold: every layer validated before any launch
    FL = lib.FoldLayer
    ok_layer = FL(0x10000, 0x10000, 0x10000, 0x10000, 1e-3, 4, 0x10000, 0x10000)
    fb = lib._lib.conv_bn_silu_fold_batch
    arr = (FL * 2)(ok_layer, FL(0x10000, None, 0x10000, 0x10000, 1e-3, 4, 0x10000, 0x10000))
    assert fb(arr, 2, None) == lib.CBS_ERR_INVALID_ARG
    arr = (FL * 2)(ok_layer, FL(0x10000, 0x10008, 0x10000, 0x10000, 1e-3, 4, 0x10000, 0x10000))
    assert fb(arr, 2, None) == lib.CBS_ERR_MISALIGNED
    arr = (FL * 1)(FL(0x10000, 0x10000, 0x10000, 0x10000, -1.0, 4, 0x10000, 0x10000))
    assert fb(arr, 1, None) == lib.CBS_ERR_INVALID_ARG
    assert fb(None, -1, None) == lib.CBS_ERR_INVALID_ARG
    assert fb(None, 0, None) == lib.CBS_OK
    arr = (FL * 1)(FL(None, None, None, None, 1e-3, 0, None, None))
    assert fb(arr, 1, None) == lib.CBS_OK                  # c_out == 0 layers are skipped
    # fold: negative eps, null pointers, misaligned, c_out == 0
    fold = lib._lib.conv_bn_silu_fold
    assert fold(good, good, good, good, -1.0, 4, good, good, None) == lib.CBS_ERR_INVALID_ARG
    assert fold(good, None, good, good, 1e-3, 4, good, good, None) == lib.CBS_ERR_INVALID_ARG
    assert fold(good, good, odd, good, 1e-3, 4, good, good, None) == lib.CBS_ERR_MISALIGNED
    assert fold(None, None, None, None, 1e-3, 0, None, None, None) == lib.CBS_OK
    assert fold(good, good, good, good, float("nan"), 4, good, good, None) == lib.CBS_ERR_INVALID_ARG


def test_status_strings(lib):
    for st in range(6):
        assert isinstance(lib._status_string(st), bytes) and lib._status_string(st)
    assert lib._status_string(99) == b"unknown status"


def test_plan_request_overrides(lib):
    """Planner overrides: each forced choice shows in the plan, and combinations the
    kernels cannot run are refused before anything launches."""
    deep = (32, 20, 20, 512, 512, 3, 3, 1, 1)
    assert lib.plan_request(*deep)["cluster"] == 2                       # the planner's own choice
    p = lib.plan_request(*deep, pair=0)
    assert p["cluster"] == 1 and p["stream_k"] == 1 and p["threads"] == 384
    p = lib.plan_request(*deep, stream_k=0)
    assert p["stream_k"] == 0 and p["cluster"] == 1 and p["workspace_bytes"] == 0
    p = lib.plan_request(*deep, block_n=128, stream_k=0)
    assert p["block_n"] == 128 and p["tiles"] == 400
    down = (16, 160, 160, 64, 128, 3, 3, 2, 1)
    assert lib.plan_request(*down)["swap_ab"] == 1
    p = lib.plan_request(*down, swap_ab=0)
    assert p["swap_ab"] == 0 and p["block_n"] == 128
    assert lib.plan_request(*down, algo="direct")["algo"] == "direct"
    for bad in ({"swap_ab": 1, "stream_k": 1}, {"swap_ab": 1, "block_n": 128}, {"pair": 1, "stream_k": 0},
                {"algo": "direct", "swap_ab": 0}):
        with pytest.raises(lib.CbsError):
            lib.plan_request(*down, **bad)
    with pytest.raises(lib.CbsError):                                     # stream-K shares < one tile
        lib.plan_request(1, 32, 32, 16, 32, 3, 3, 1, 1, stream_k=1)
    with pytest.raises(lib.CbsError):                                     # thin-input kernel: no tilings
        lib.plan_request(1, 640, 640, 3, 16, 3, 3, 2, 1, swap_ab=0)
    for bad in ({"swap_ab": 2}, {"pair": -2}, {"block_n": 48}, {"wait_timeout_ns": -1}, {"balanced": 2}):
        with pytest.raises(lib.CbsError) as e:
            lib.plan_request(*down, **bad)
        assert e.value.status == lib.CBS_ERR_INVALID_ARG


def test_balanced_channel_major_plans(lib):
    """Channel-major (swap AB) plans deal equal runs of 32-pixel chunks by default; whole
    256-pixel tiles on request; a balanced run is refused on pixel-major tiles."""
    pointwise = (16, 40, 40, 256, 256, 1, 1, 1, 0)   # 200 whole tiles: 48 CTAs would take two
    p = lib.plan_request(*pointwise, row_boxes=0)      # the tc_conv.cu channel-major kernel
    assert p["swap_ab"] == 1 and p["balanced"] == 1 and p["grid"] == 152 and p["row_boxes"] == 0
    p0 = lib.plan_request(*pointwise, balanced=0)
    assert p0["swap_ab"] == 1 and p0["balanced"] == 0 and p0["grid"] == 152 and p0["tiles"] == 200
    assert lib.plan(*pointwise)["row_boxes"] == 1
    tiny_swap = (2, 13, 11, 16, 24, 3, 3, 1, 1)      # 286 pixels: 9 chunks, so 9 CTAs
    assert lib.plan_request(*tiny_swap, swap_ab=1, row_boxes=0)["grid"] == 9
    assert lib.plan_request(*tiny_swap, swap_ab=1, balanced=0)["grid"] == 2
    deep = (32, 20, 20, 512, 512, 3, 3, 1, 1)
    assert lib.plan_request(*deep)["balanced"] == 0
    assert lib.plan_request(*deep, balanced=0)["balanced"] == 0
    with pytest.raises(lib.CbsError) as e:
        lib.plan_request(*deep, balanced=1)
    assert e.value.status == lib.CBS_ERR_UNSUPPORTED


def test_tuning_sweep_variants_are_consistent():
    from conv2d_batchnorm_silu_gb300 import tune
    vs = list(tune.variants())
    labels = [v[0] for v in vs]
    assert len(labels) == len(set(labels)) and labels[:2] == ["auto", "direct"]
    for label, ov in vs[2:]:
        if "row_boxes" in ov and "swap_ab" not in ov:   # the channel-major kernel of tc_cmajor.cu
            assert ov["row_boxes"] in (0, 1) and ov["weights_resident"] in (0, 1)
            assert ov["row_boxes"] or ov["weights_resident"]
            continue
        assert not (ov["pair"] and not ov["stream_k"])
        assert not (ov["swap_ab"] and (ov["stream_k"] or ov["pair"]))
        assert ov.get("balanced", -1) != 1 or ov["swap_ab"] == 1
    assert len(tune.SWEEP) >= 15 and len({s.name for s in tune.SWEEP}) == len(tune.SWEEP)



def test_planner_choices_match_the_measured_sweep():
    """The planner's choice for every layer of the threshold sweep (tune.SWEEP) on a
    152-SM GB300, as the committed planner sweep (tune.py on a GB300) measured
    it: a change to the planner's rules changes one of these and calls for the sweep to
    be run again."""
    from conv2d_batchnorm_silu_gb300 import capi, tune
    expected = {
        "stem640": "thin-input", "down320": "wres", "c2f160_1x1": "rows", "bneck160": "wres",
        "down160": "swap", "c2f80_1x1": "rows", "bneck80": "swap", "down80": "swap",
        "c2f40_1x1": "rows", "bneck40": "swap", "down40": "swap", "c2f20_1x1": "rows",
        "bneck20": "swap", "sppf20_1x1": "rows", "head80_3x3": "swap", "tiny": "n32",
        "stem": "thin-input", "down": "rows", "pointwise": "rows", "deep": "n256-sk-pair",
    }
    got = {}
    for sh in tune.SWEEP:
        p = capi.plan(sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad, "auto", 152)
        got[sh.name] = tune._plan_label(p)
    assert got == expected


def test_noalloc_fallback_plan_needs_no_scratch(lib):
    """conv_bn_silu_forward_noalloc holds 20 MiB of stream-K scratch.  On a 152-SM GB300
    every stream-K split fits; with more SMs a split can need more, and the entry point
    then runs the whole-tile plan (stream_k = 0, pair = 0), which must exist and need none."""
    cap = 20 << 20
    deep = (32, 20, 20, 512, 512, 3, 3, 1, 1)
    split244 = (39, 20, 20, 256, 384, 3, 3, 1, 1)
    for shape in (deep, split244):
        assert lib.plan_request(*shape, sm_count=152)["workspace_bytes"] <= cap
    over = 0
    for sms in (160, 170, 188, 200):
        for shape in (deep, split244):
            p = lib.plan_request(*shape, sm_count=sms)
            if p["stream_k"] and p["workspace_bytes"] > cap:
                over += 1
                q = lib.plan_request(*shape, sm_count=sms, stream_k=0, pair=0)
                assert q["stream_k"] == 0 and q["cluster"] == 1 and q["workspace_bytes"] == 0
    assert over > 0   # the fallback is reachable on some larger GPU
