"""C ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments with the documented codes before
touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

import attention_attn_fwd_gb300 as attn
from attention_attn_fwd_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return attn.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_status_string", "attn_device_status",
              "attn_tile_config", "attn_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", attn.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line)
    for name in declared_functions():
        assert name in exported, name


def test_status_strings(lib):
    for code in range(6):
        s = attn.attn_status_string(code)
        assert s and s != "unknown status"
    assert attn.attn_status_string(99) == "unknown status"


def test_version(lib):
    assert attn.attn_version() >= 100


BAD = 0x1000  # an aligned address that is never dereferenced on these paths


def call(**kw):
    a = dict(Q=BAD, K=BAD + 0x100000, V=BAD + 0x200000, O=BAD + 0x300000,
             LSE=0, B=1, Hq=2, Hkv=2, Sq=128, Skv=128, D=64, scale=0.125,
             causal=0, input_pos=0, dtype=attn.ATTN_F16, stream=0)
    a.update(kw)
    return attn.attn_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=3, Hkv=2), attn.ATTN_ERR_INVALID_ARG),       # Hq % Hkv
    (dict(Hq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Sq=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Skv=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(input_pos=-1, causal=1), attn.ATTN_ERR_INVALID_ARG),
    (dict(input_pos=2**31 - 100, Sq=128), attn.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Q=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(O=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Q=BAD + 8), attn.ATTN_ERR_ALIGNMENT),
    (dict(V=BAD + 0x200002), attn.ATTN_ERR_ALIGNMENT),
    (dict(LSE=BAD + 0x400002), attn.ATTN_ERR_ALIGNMENT),
    (dict(O=BAD + 0x40), attn.ATTN_ERR_INVALID_ARG),       # O overlaps Q
])
def test_argument_checks(lib, kw, code):
    assert call(**kw) == code


def test_empty_problem_is_a_noop(lib):
    assert call(B=0) == attn.ATTN_OK
    assert call(Sq=0) == attn.ATTN_OK
    # Even with NULL pointers: nothing is read or written.
    assert call(Sq=0, Q=0, K=0, V=0, O=0) == attn.ATTN_OK


def test_tile_config(lib):
    c = attn.attn_tile_config(1, 32, 4, 8192, 8192, 128, 1, 0, attn.ATTN_BF16)
    assert c["block_m"] == 256 and c["block_n"] == 128
    assert c["grid"] == 32 * 8192 // 256
    assert 0 < c["smem_bytes"] <= 227 * 1024
    assert c["stages"] >= 2
    c64 = attn.attn_tile_config(4, 16, 16, 1000, 1000, 64, 0, 0, attn.ATTN_F16)
    assert c64["grid"] == 4 * 16 * 4
    # Decode shape: the 4 query heads of each K/V head share one tile.
    cd = attn.attn_tile_config(8, 32, 8, 1, 4096, 128, 1, 4095, attn.ATTN_BF16)
    assert cd["block_m"] == 4 and cd["grid"] == 8 * 8
    with pytest.raises(attn.AttnError):
        attn.attn_tile_config(1, 3, 2, 8, 8, 64, 0, 0, attn.ATTN_F16)


def test_splitkv_plan_host_only(lib):
    """An explicit split request is planned without a GPU."""
    ns, ws = attn.attn_splitkv_plan(2, 8, 2, 1, 1000, 128, 1, 999,
                                    attn.ATTN_BF16, 5)
    assert ns == 4           # 8 tiles in 5 requested ranges: 2 tiles each
    rows = 2 * 8 * 1
    # fp32 partial outputs, then fp32 partial LSEs, each 256-byte aligned.
    assert ws == (-(-(ns * rows * 128 * 4) // 256) * 256 +
                  -(-(ns * rows * 4) // 256) * 256)
    ns1, _ = attn.attn_splitkv_plan(1, 2, 2, 4, 100, 64, 0, 0,
                                    attn.ATTN_F16, 8)
    assert ns1 == 1          # 100 keys: a single tile
    with pytest.raises(attn.AttnError):
        attn.attn_splitkv_plan(1, 3, 2, 4, 100, 64, 0, 0, attn.ATTN_F16, 2)


# (B, Hq, Hkv, Sq, Skv, D, causal, input_pos) and the automatic split count
# on 152 SMs; each was the best or within 5 % of the best measured count on
# a GB300 over 1-32 ranges (bf16).
PLAN_PICKS = [
    ((8, 32, 8, 1, 4096, 128, 1, 4095), 2),          # decode: clusters of 2
    ((4, 32, 8, 16, 16384, 128, 1, 16368), 4),       # packed chunk: clusters
    ((1, 32, 8, 512, 32768, 128, 1, 32256), 2),      # one wave of 128 units
    ((2, 16, 16, 1024, 16384, 128, 1, 15360), 1),    # one pass fills the GPU
    ((1, 8, 8, 128, 131072, 128, 1, 130944), 16),    # bound by K/V streaming
    ((1, 8, 8, 256, 32768, 128, 1, 32512), 19),      # one wave of 152 units
    ((1, 16, 16, 256, 32768, 64, 1, 32512), 9),      # D = 64, one wave
]


@pytest.mark.parametrize("shape, expect", PLAN_PICKS)
def test_splitkv_plan_auto_host(lib, shape, expect):
    """The automatic count is planned on the host (152 SMs without a
    device), and only counts attn_fwd_splitkv accepts come out."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the device's SM count applies")
    ns, ws = attn.attn_splitkv_plan(*shape, attn.ATTN_BF16, 0)
    assert ns == expect
    assert attn.attn_splitkv_plan(*shape, attn.ATTN_BF16, ns) == (ns, ws)


def test_splitkv_argument_checks(lib):
    a = dict(Q=BAD, K=BAD + 0x100000, V=BAD + 0x200000, O=BAD + 0x300000,
             LSE=0, B=1, Hq=2, Hkv=2, Sq=1, Skv=1000, D=128, scale=0.1,
             causal=1, input_pos=999, dtype=attn.ATTN_BF16, num_splits=2,
             workspace=BAD + 0x400000, workspace_bytes=1 << 20, stream=0)
    assert attn.attn_fwd_splitkv(**dict(a, num_splits=0)) == \
        attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_splitkv(**dict(a, num_splits=500)) == \
        attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_splitkv(**dict(a, D=80)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_fwd_splitkv(**dict(a, Sq=0)) == attn.ATTN_OK


def test_no_device_is_an_error_not_a_crash(lib):
    """Without a GPU a well-formed call fails cleanly with ATTN_ERR_CUDA or
    ATTN_ERR_INVALID_ARG (pointers are not device memory)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call() in (attn.ATTN_ERR_CUDA, attn.ATTN_ERR_INVALID_ARG)


def test_fwd_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(attn.AttnError):
        attn.fwd(q, q, q)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(attn, "_LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(attn, "_lib", None)
    with pytest.raises(attn.AttnError, match="not built"):
        attn.load_library()


def test_fp8_tile_config_and_plan(lib):
    """E4M3 inputs: 128-byte rows at D = 128 give 16 KB tiles (twice the
    ring slots of bf16 at D = 128); D = 64 is not implemented."""
    c8 = attn.attn_tile_config(1, 32, 4, 8192, 8192, 128, 1, 0, attn.ATTN_E4M3)
    c16 = attn.attn_tile_config(1, 32, 4, 8192, 8192, 128, 1, 0,
                                attn.ATTN_BF16)
    assert c8["block_m"] == c16["block_m"] and c8["grid"] == c16["grid"]
    assert c8["stages"] == 2 * c16["stages"]
    assert c8["smem_bytes"] < c16["smem_bytes"]
    with pytest.raises(attn.AttnError):
        attn.attn_tile_config(1, 2, 2, 128, 128, 64, 0, 0, attn.ATTN_E4M3)
    ns, ws = attn.attn_splitkv_plan(2, 8, 2, 1, 1000, 128, 1, 999,
                                    attn.ATTN_E4M3, 5)
    assert (ns, ws) == attn.attn_splitkv_plan(2, 8, 2, 1, 1000, 128, 1, 999,
                                              attn.ATTN_BF16, 5)


def fp8_call(**kw):
    a = dict(Q=BAD, K=BAD + 0x100000, V=BAD + 0x200000, O=BAD + 0x300000,
             LSE=0, B=1, Hq=2, Hkv=2, Sq=128, Skv=128, D=128, scale=0.125,
             q_descale=1.0, k_descale=1.0, v_descale=1.0, causal=0,
             input_pos=0, window=0, num_splits=0, workspace=0,
             workspace_bytes=0, stream=0)
    a.update(kw)
    return attn.attn_fwd_fp8(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q_descale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(k_descale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(v_descale=float("-inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=1e30, q_descale=1e30), attn.ATTN_ERR_INVALID_ARG),
    (dict(num_splits=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(window=4), attn.ATTN_ERR_INVALID_ARG),          # window, no causal
    (dict(Q=BAD + 8), attn.ATTN_ERR_ALIGNMENT),
    (dict(Sq=0), attn.ATTN_OK),
    (dict(B=0, Q=0, K=0, V=0, O=0), attn.ATTN_OK),
])
def test_fp8_argument_checks(lib, kw, code):
    assert fp8_call(**kw) == code


def test_e4m3_refused_by_16_bit_entry_points(lib):
    assert call(dtype=attn.ATTN_E4M3, D=128) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_window(BAD, BAD + 0x100000, BAD + 0x200000,
                                BAD + 0x300000, 0, 1, 2, 2, 128, 128, 128,
                                0.1, 1, 0, 0, attn.ATTN_E4M3, 0) == \
        attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_splitkv(BAD, BAD + 0x100000, BAD + 0x200000,
                                 BAD + 0x300000, 0, 1, 2, 2, 1, 1000, 128,
                                 0.1, 1, 999, attn.ATTN_E4M3, 2,
                                 BAD + 0x400000, 1 << 20, 0) == \
        attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd(BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, BAD, 1, 2,
                         2, 128, 128, 128, 0.1, 1, 0, 0, attn.ATTN_E4M3,
                         BAD, 1 << 20, 0) == attn.ATTN_ERR_UNSUPPORTED


def test_bwd_workspace_bytes(lib):
    """Two fp32 vectors (lse2 and D) per query row, each row plane padded
    to whole 128-row tiles, each vector rounded up to 256 bytes; 0 for
    negative sizes (the documented contract of attn_bwd_workspace_bytes)."""
    def expect(B, Hq, Sq):
        rows = B * Hq * (-(-Sq // 128) * 128)
        return 2 * (-(-(rows * 4) // 256) * 256)

    for B, Hq, Sq in [(1, 2, 64), (1, 2, 128), (1, 2, 129), (2, 32, 8192),
                      (3, 5, 1), (1, 1, 0), (0, 4, 100)]:
        assert attn.attn_bwd_workspace_bytes(B, Hq, Sq) == expect(B, Hq, Sq)
    for bad in [(-1, 2, 64), (1, -2, 64), (1, 2, -64)]:
        assert attn.attn_bwd_workspace_bytes(*bad) == 0
    # Padding: every Sq in one 128-row tile needs the same workspace.
    assert len({attn.attn_bwd_workspace_bytes(1, 4, s)
                for s in range(1, 129)}) == 1


def test_dispatch_entries_host_only(lib):
    """attn_dispatch names the table entry without a GPU: tile mode, unit
    order and O store follow the group size, Sq, the mask and the split
    count; bad arguments get the validation code attn_fwd would return."""
    bf, f16, e4 = attn.ATTN_BF16, attn.ATTN_F16, attn.ATTN_E4M3
    e = attn.attn_dispatch(1, 32, 4, 8192, 8192, 128, 1, 0, bf)
    assert e["name"] == "d128.bf16.paired-heads.plan.tma"
    assert (e["q_tiles"], e["paired"], e["s_buffers"], e["order"],
            e["o_store"], e["hold_scores"], e["num_splits"]) == \
        (2, 1, 2, 2, 1, 1, 0)
    assert e["units"] == 32 // 2 * 8192 // 128
    # The plan's unit bound makes the causal entry depend on Sq: 2048
    # units at 16k keep the LPT rounds, as do fewer units than SMs.
    e = attn.attn_dispatch(1, 32, 4, 16384, 16384, 128, 1, 0, bf)
    assert e["name"] == "d128.bf16.paired-heads.lpt.tma" and e["order"] == 0
    e = attn.attn_dispatch(1, 32, 4, 1024, 1024, 128, 1, 0, bf)
    assert e["order"] == 0 and e["units"] == 128
    e = attn.attn_dispatch(1, 32, 32, 4096, 4096, 128, 1, 0, f16)
    assert e["name"] == "d128.f16.256-rows.plan.tma"
    e = attn.attn_dispatch(4, 16, 16, 1024, 1024, 64, 0, 0, f16)
    assert e["name"] == "d64.f16.256-rows.head-major.tma"
    assert e["s_buffers"] == 3 and e["units"] == 4 * 16 * 4
    e = attn.attn_dispatch(8, 32, 8, 1, 4096, 128, 1, 4095, bf, num_splits=2)
    assert e["name"] == "d128.bf16.gqa-packed.lpt.rows"
    assert e["q_tiles"] == 1 and e["num_splits"] == 2
    assert e["units"] == 8 * 8 * 2 and e["block_m"] == 4
    # Merge modes: the decode's 128 units fit the SMs, 2 ranges per
    # cluster; 4 ranges are 256 units (more than the 152 SMs),
    # and unpacked tiles always merge in the second kernel.
    assert e["merge"] == 1
    e = attn.attn_dispatch(8, 32, 8, 1, 4096, 128, 1, 4095, bf, num_splits=4)
    assert e["merge"] == 2 and e["units"] == 8 * 8 * 4
    e = attn.attn_dispatch(1, 8, 8, 256, 32768, 128, 1, 32512, bf,
                           num_splits=8)
    assert e["merge"] == 2 and e["q_tiles"] == 2
    assert attn.attn_dispatch(1, 8, 8, 256, 32768, 128, 1, 32512,
                              bf)["merge"] == 0
    e = attn.attn_dispatch(1, 32, 4, 8192, 8192, 128, 1, 0, e4)
    assert e["name"] == "d128.e4m3.paired-heads.plan.tma"
    # window entry: causal, LPT order
    e = attn.attn_dispatch(1, 32, 4, 32768, 32768, 128, 1, 0, bf,
                           window=4096)
    assert e["order"] == 0
    for bad in [dict(Hq=3, Hkv=2), dict(D=96), dict(window=8, causal=0)]:
        args = dict(B=1, Hq=2, Hkv=2, Sq=64, Skv=64, D=64, causal=1,
                    input_pos=0, dtype=f16)
        args.update(bad)
        with pytest.raises(attn.AttnError):
            attn.attn_dispatch(args["B"], args["Hq"], args["Hkv"], args["Sq"],
                               args["Skv"], args["D"], args["causal"],
                               args["input_pos"], args["dtype"],
                               window=args.get("window", 0))
