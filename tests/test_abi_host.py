"""The C-ABI library loads and exports every symbol include/fp8g.h declares,
and rejects invalid arguments on the host before touching the GPU.  No
compute call is made (these tests also run where no GPU exists)."""
import ctypes
import os
import re

import pytest

import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
from fp8_tensor_core_gb300 import _lib
from fp8_tensor_core_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8g.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    for n in ("fp8_gemm_nt", "fp8_gemm_grouped_masked", "fp8g_get_device_status",
              "fp8g_status_string", "fp8g_version", "fp8g_set_wait_timeout_ns"):
        assert n in names
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    names = [lib.fp8g_status_string(i).decode() for i in range(8)]
    assert names[0] == "FP8G_OK" and names[5] == "FP8G_ERR_TIMEOUT"
    assert len(set(names)) == 8
    assert lib.fp8g_status_string(99).decode() == "FP8G_UNKNOWN_STATUS"
    assert lib.fp8g_version() >= 100


def test_timeout_setting_roundtrip(lib):
    prev = lib.fp8g_set_wait_timeout_ns(12345)
    assert lib.fp8g_set_wait_timeout_ns(0) == 12345
    assert lib.fp8g_set_wait_timeout_ns(prev) == 2_000_000_000


ALIGNED = 0x10000   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args,code", [
    ((0, ALIGNED, ALIGNED, 16, 16, 16, 0, 0, 0), 1),        # null A
    ((ALIGNED, ALIGNED, 0, 16, 16, 16, 0, 0, 0), 1),        # null D
    ((ALIGNED, ALIGNED, ALIGNED, 0, 16, 16, 0, 0, 0), 1),   # M = 0
    ((ALIGNED, ALIGNED, ALIGNED, 16, 16, 24, 0, 0, 0), 1),  # K % 16
    ((ALIGNED, ALIGNED, ALIGNED, 16, 12, 16, 0, 0, 0), 1),  # N % 8
    ((ALIGNED, ALIGNED, ALIGNED, 16, 16, 16, 2, 0, 0), 1),  # bad dtype
    ((ALIGNED, ALIGNED, ALIGNED, 16, 16, -16, 0, 0, 0), 1), # negative K
    ((ALIGNED, ALIGNED, ALIGNED, 1 << 31, 16, 16, 0, 0, 0), 1),  # M too large
    ((ALIGNED + 8, ALIGNED, ALIGNED, 16, 16, 16, 0, 0, 0), 2),  # misaligned A
    ((ALIGNED, ALIGNED, ALIGNED + 2, 16, 16, 16, 0, 0, 0), 2),  # misaligned D
])
def test_dense_validation(lib, args, code):
    assert lib.fp8_gemm_nt(*args, None) == code


@pytest.mark.parametrize("args,code", [
    ((ALIGNED, ALIGNED, ALIGNED, 0, 4, 64, 64, 64, 0, 0, 0, 0), 1),        # null masked_m
    ((ALIGNED, ALIGNED, ALIGNED, ALIGNED, 0, 64, 64, 64, 0, 0, 0, 0), 1),  # G = 0
    ((ALIGNED, ALIGNED, ALIGNED, ALIGNED, 4, 64, 64, 64, 65, 0, 0, 0), 1), # hint > M_max
    ((ALIGNED, ALIGNED, ALIGNED, ALIGNED, 4, 64, 64, 64, -1, 0, 0, 0), 1), # hint < 0
    ((ALIGNED, ALIGNED, ALIGNED, ALIGNED, 2048, 64, 64, 64, 0, 0, 0, 0), 3),  # too many groups
    ((ALIGNED, ALIGNED, ALIGNED, ALIGNED + 4, 4, 64, 64, 64, 0, 0, 0, 0), 2), # masked_m misaligned
    ((ALIGNED, ALIGNED, ALIGNED, ALIGNED, 4, 64, 60, 64, 0, 0, 0, 0), 1),  # N % 8
])
def test_grouped_validation(lib, args, code):
    assert lib.fp8_gemm_grouped_masked(*args, None) == code


def test_invalid_swap_mode(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("would reach the device with fake pointers")
    # without a device the call stops at device discovery
    assert lib.fp8_gemm_nt(ALIGNED, ALIGNED, ALIGNED, 16, 16, 16, 0, 0, 0, None) == 6


def test_get_device_status_rejects_null(lib):
    assert lib.fp8g_get_device_status(None, None) == 1


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    import fp8_tensor_core_gb300 as fp8g
    a = torch.zeros((16, 16), dtype=torch.uint8)
    with pytest.raises(ValueError):
        fp8g.fp8_gemm_nt(a, a, a_dtype=0, b_dtype=0)


def test_python_flag_constants_match_the_header():
    """Every flag the binding exports has the value the C header defines."""
    import re
    import fp8_tensor_core_gb300 as fp8g
    with open(os.path.join(ROOT, "include", "fp8g.h")) as f:
        defs = dict(re.findall(r"#define FP8G_([A-Z0-9_]+) (0x[0-9a-fA-F]+|[0-9]+)u?\b", f.read()))
    checked = 0
    for name in ("SWAP_AUTO", "SWAP_ON", "SWAP_OFF", "DEBUG_ONE_STAGE", "WHOLE_TILES", "STREAM_K", "SINGLE_SM_TILES",
                 "NO_PDL", "PAIR_TILES", "ONE_MMA_ISSUER", "TWO_MMA_ISSUERS", "SHARE_SM", "NO_SHARE_SM", "SPLIT_TAIL"):
        assert name in defs, name
        assert getattr(fp8g, name) == int(defs[name], 0), name
        checked += 1
    assert checked == 14


def test_field_flags_do_not_overlap_the_single_bit_flags():
    """STAGES, TILE_N and TOKEN_BOX fill their own bit fields and leave every
    single-bit flag alone."""
    import fp8_tensor_core_gb300 as fp8g
    singles = 0
    for name in ("SWAP_ON", "SWAP_OFF", "DEBUG_ONE_STAGE", "WHOLE_TILES", "STREAM_K", "SINGLE_SM_TILES", "NO_PDL",
                 "PAIR_TILES", "ONE_MMA_ISSUER", "TWO_MMA_ISSUERS", "SHARE_SM", "NO_SHARE_SM", "SPLIT_TAIL"):
        assert singles & getattr(fp8g, name) == 0, name
        singles |= getattr(fp8g, name)
    fields = [fp8g.STAGES(15), fp8g.TILE_N(15 * 32), fp8g.TOKEN_BOX(15 * 16)]
    for i, f in enumerate(fields):
        assert f & singles == 0
        for g in fields[i + 1:]:
            assert f & g == 0
    assert fp8g.TOKEN_BOX(48) == 3 << 24 and fp8g.TOKEN_BOX(0) == 0



# ---- the plan query (no device needed when the device is described) ------------------

GB300 = dict(sms=152, smem_optin=232448)


def _plan(layout, G, rows, N, K, hint=0, sf=0, flags=0):
    import fp8_tensor_core_gb300 as fp8g
    return fp8g.fp8g_describe_plan(layout, G, rows, N, K, hint, sf, flags, **GB300)


@pytest.mark.parametrize("args,expect", [
    # dense 4096^3: SM-pair tiles 256 wide, three whole waves and the last 28
    # tiles split two ways along K; the 8192-row projections: the 18432 x 7168
    # one splits its last 24 tiles three ways, 7168 x 18432 (60 left) none
    ((0, 1, 4096, 4096, 4096), dict(kernel=1, tile_n=256, stream_k=1, k_split=2, grid=152)),
    ((0, 1, 8192, 18432, 7168), dict(kernel=1, tile_n=256, k_split=3)),
    ((0, 1, 8192, 7168, 18432), dict(kernel=1, tile_n=256, k_split=1, stream_k=0)),
    # small-M weight streaming: token tiles at N=24576, K=1536 (A box of the one row) ...
    ((0, 1, 1, 24576, 1536), dict(kernel=0, tile_n=192, token_box=1, grid=128)),
    ((0, 1, 33, 24576, 1536), dict(kernel=0, token_box=33)),
    # ... SwapAB stream-K at N=7168, K=16384, sharing the SM up to 16 tokens
    ((0, 1, 16, 7168, 16384), dict(kernel=2, tile_n=16, stream_k=1, shared_sm=1, token_box=16, grid=152)),
    ((0, 1, 5, 7168, 16384), dict(kernel=2, tile_n=16, shared_sm=1, token_box=5)),
    ((0, 1, 64, 7168, 16384), dict(kernel=2, tile_n=64, shared_sm=0, token_box=64)),
    # masked MoE decode (32 experts, up to 32 tokens): token tiles; forced SwapAB: 16-row boxes
    ((1, 32, 128, 4096, 7168, 32), dict(kernel=0)),
    ((1, 32, 128, 4096, 7168, 32, 0, 1), dict(kernel=2, tile_n=32, token_box=16, stream_k=1)),
    # 16 experts: SwapAB at 160 tokens for N=4096, K=7168, token tiles at 96 and for N=7168, K=2048
    ((1, 16, 160, 4096, 7168, 160), dict(kernel=2, tile_n=160, token_box=160)),
    ((1, 16, 96, 4096, 7168, 96), dict(kernel=0)),
    ((1, 16, 160, 7168, 2048, 160), dict(kernel=0)),
    # contiguous groups of 256 tokens: SM pairs
    ((2, 32, 8192, 4096, 7168), dict(kernel=1, tile_n=256)),
    # block scales: single-SM tiles 224 wide (256 wide from 48 K blocks); SwapAB with two issuers
    ((0, 1, 4096, 4096, 4096, 0, 128), dict(kernel=0, tile_n=224, mma_issuers=1)),
    ((0, 1, 8192, 7168, 18432, 0, 128), dict(kernel=0, tile_n=256)),
    ((1, 32, 128, 4096, 7168, 32, 128, 1), dict(kernel=2, tile_n=32, token_box=32, mma_issuers=2)),
])
def test_describe_plan_pins_the_automatic_choices(args, expect):
    got = _plan(*args)
    assert {k: got[k] for k in expect} == expect, got
    assert got["stages"] >= 1 and 1 <= got["grid"] <= 152
    if got["mma_issuers"] == 2:
        assert got["stages"] % 2 == 0


def test_describe_plan_follows_the_flags():
    import fp8_tensor_core_gb300 as fp8g
    assert _plan(0, 1, 16, 7168, 16384, flags=fp8g.NO_SHARE_SM)["shared_sm"] == 0
    assert _plan(0, 1, 64, 7168, 16384, flags=fp8g.SWAP_OFF)["kernel"] == 0
    assert _plan(0, 1, 4096, 4096, 4096, flags=fp8g.SINGLE_SM_TILES)["kernel"] == 0
    assert _plan(0, 1, 4096, 4096, 4096, flags=fp8g.TILE_N(224))["tile_n"] == 224
    assert _plan(0, 1, 4096, 4096, 4096, flags=fp8g.STAGES(3))["stages"] == 3
    assert _plan(0, 1, 128, 4096, 4096, flags=fp8g.SWAP_ON | fp8g.TOKEN_BOX(32))["token_box"] == 32
    assert _plan(0, 1, 64, 7168, 16384, flags=fp8g.WHOLE_TILES)["stream_k"] == 0
    assert _plan(0, 1, 4096, 4096, 4096, flags=fp8g.WHOLE_TILES)["k_split"] == 1
    assert _plan(0, 1, 4096, 4096, 4096, flags=fp8g.STREAM_K)["k_split"] == 0


@pytest.mark.parametrize("args,code", [
    ((3, 1, 16, 4096, 4096, 0, 0, 0, 152, 232448), 1),      # no such layout
    ((0, 2, 16, 4096, 4096, 0, 0, 0, 152, 232448), 1),      # dense takes one group
    ((0, 1, 16, 4096, 4100, 0, 0, 0, 152, 232448), 1),      # K % 16
    ((0, 1, 16, 4100, 4096, 0, 0, 0, 152, 232448), 1),      # N % 8
    ((1, 4, 16, 4096, 4096, 32, 0, 0, 152, 232448), 1),     # hint above rows
    ((0, 1, 16, 4096, 4096, 0, 64, 0, 152, 232448), 1),     # group size
    ((0, 1, 16, 4096, 4096, 0, 0, 0, 152, 0), 1),           # half a device description
    ((0, 1, 16, 4096, 4096, 0, 0, 3, 152, 232448), 1),      # swap mode 3
    ((2, 4, 64, 4096, 4096, 0, 128, 0, 152, 232448), 3),    # block scales with the contiguous layout
])
def test_describe_plan_argument_errors(lib, args, code):
    out = _lib.Plan()
    assert lib.fp8g_describe_plan(*args, ctypes.byref(out)) == code
    assert lib.fp8g_describe_plan(0, 1, 16, 4096, 4096, 0, 0, 0, 152, 232448, None) == 1


def test_plan_struct_matches_the_header():
    """The binding's fp8g_plan fields are the header's, in order, all int32."""
    src = open(HEADER).read()
    body = re.search(r"typedef struct fp8g_plan \{(.*?)\} fp8g_plan;", src, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"int32_t\s+([a-z_]+);", body)
    assert fields == [name for name, _ in _lib.Plan._fields_]
    assert ctypes.sizeof(_lib.Plan) == 4 * len(fields)
    import fp8_tensor_core_gb300 as fp8g
    defs = dict(re.findall(r"#define FP8G_KERNEL_([A-Z_]+) ([0-9]+)", src))
    assert (int(defs["TOKEN_TILES"]), int(defs["SM_PAIRS"]), int(defs["SWAP_AB"])) == \
        (fp8g.KERNEL_TOKEN_TILES, fp8g.KERNEL_SM_PAIRS, fp8g.KERNEL_SWAP_AB)
