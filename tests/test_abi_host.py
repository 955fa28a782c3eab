"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/fa.h declares; argument checks that return before any device
work.  No compute call is made here (this runs without a GPU)."""
import ctypes
import os
import re

import pytest

from exact_attention_76_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_expected_entry_points():
    syms = declared_symbols()
    for name in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_fwd_fp8", "fa_status_string",
                 "fa_device_error", "fa_bwd_preprocess", "fa_bwd_main", "fa_bwd_dq_convert"):
        assert name in syms
    assert set(syms) == set(_lib.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_lib.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code in range(8):
        s = lib.fa_status_string(code).decode()
        assert s.startswith(_lib.STATUS_NAMES[code])


def test_workspace_size(lib):
    B, H, N, d = 2, 3, 130, 64
    rows = B * H * N
    expect = ((rows * 4 + 15) // 16) * 16 + rows * d * 4
    assert lib.fa_bwd_workspace_size(B, H, N, d) == expect
    assert lib.fa_bwd_workspace_size(1, 1, 1, 96) == 0
    assert lib.fa_bwd_workspace_size(0, 1, 1, 64) == 0


def _grouped_decode_chunks(B, Hkv, N):
    """Chunks per (batch, key/value head) of the grouped decode: one resident
    wave of two CTAs per SM on 152 SMs while B*Hkv is below it, else the split
    (1..4) with the fewest waves per unit of work; chunks whole 128-key tiles."""
    wave, units, tiles = 2 * 152, B * Hkv, -(-N // 128)
    if units < wave:
        ns = wave // units
    else:
        ns = min(range(1, 5), key=lambda c: (-(-(units * c) // wave) / c, c))
    ns = max(1, min(ns, tiles))
    chunk = -(-(-(-N // ns)) // 128) * 128
    return -(-N // chunk)


@pytest.mark.parametrize("B,H,Hkv,N,d,chunks", [
    (1, 32, 8, 131072, 128, 38),   # 8 key/value heads: 304 CTAs, one wave
    (8, 32, 8, 8192, 128, 4),      # 64 heads x 4 chunks of 2048 keys
    (32, 64, 8, 4096, 128, 1),     # 256 heads: one chunk each
    (32, 32, 16, 4096, 64, 4),     # 512 heads: 2048 CTAs in 7 waves beat 1 to 3 chunks
    (2, 4, 2, 63, 64, 1),          # fewer keys than a tile
])
def test_grouped_decode_workspace_follows_the_chunk_plan(lib, B, H, Hkv, N, d, chunks):
    assert _grouped_decode_chunks(B, Hkv, N) == chunks
    assert lib.fa_decode_workspace_size(B, H, Hkv, N, d) == B * H * chunks * (d + 4) * 4


def test_gqa_workspace_size(lib):
    # room for the fp32 dK and dV accumulators only for groups of four query
    # heads or more, or when the key/value heads give fewer than two waves of
    # per-key/value-head CTAs on 152 SMs
    base = lib.fa_bwd_workspace_size(2, 32, 8192, 128)
    assert lib.fa_bwd_gqa_workspace_size(2, 32, 32, 8192, 128) == base          # every head its own
    assert lib.fa_bwd_gqa_workspace_size(2, 32, 16, 8192, 128) == base          # groups of 2, 2048 CTAs
    assert lib.fa_bwd_gqa_workspace_size(2, 32, 8, 8192, 128) == base + 2 * 2 * 8 * 8192 * 128 * 4  # groups of 4
    assert lib.fa_bwd_gqa_workspace_size(2, 32, 1, 8192, 128) == base + 2 * 2 * 1 * 8192 * 128 * 4  # 128 CTAs
    assert lib.fa_bwd_gqa_workspace_size(1, 4, 2, 128, 64) == lib.fa_bwd_workspace_size(1, 4, 128, 64) + 2 * 2 * 128 * 64 * 4  # 2 CTAs
    assert lib.fa_bwd_gqa_workspace_size(2, 32, 3, 8192, 128) == 0             # 3 does not divide 32
    assert lib.fa_bwd_gqa_workspace_size(2, 4, 1, 1, 64) == lib.fa_bwd_workspace_size(2, 4, 1, 64) + 2 * 2 * 64 * 4


ALIGNED = 0x10000


def fwd(lib, q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=ALIGNED, B=1, H=1, N=128, d=64, causal=0,
        scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def test_fwd_argument_errors_before_any_launch(lib):
    assert fwd(lib, q=None) == 1
    assert fwd(lib, lse=None) == 1
    assert fwd(lib, k=ALIGNED + 8) == 3
    assert fwd(lib, N=0) == 1
    assert fwd(lib, B=-1) == 1
    assert fwd(lib, d=96) == 2
    assert fwd(lib, d=256) == 2
    assert fwd(lib, scale=float("nan")) == 1
    assert fwd(lib, scale=0.0) == 1
    assert fwd(lib, scale=-1.0) == 1
    assert fwd(lib, causal=2) == 1


def test_bwd_argument_errors_before_any_launch(lib):
    p = ALIGNED
    args = [p] * 10 + [10 ** 9, 1, 1, 128, 64, 0, 0.125, None]
    assert lib.fa_bwd(*args[:9], None, *args[10:]) == 6      # no workspace
    small = list(args); small[10] = 16
    assert lib.fa_bwd(*small) == 6                            # too small
    mis = list(args); mis[9] = p + 4
    assert lib.fa_bwd(*mis) == 3                              # misaligned workspace
    nul = list(args); nul[6] = None
    assert lib.fa_bwd(*nul) == 1


def test_fp8_argument_errors_before_any_launch(lib):
    p = ALIGNED
    assert lib.fa_fwd_fp8(p, p, p, None, p, p, p, p, 1, 1, 128, 128, 0, 0.1, None) == 1
    assert lib.fa_fwd_fp8(p, p, p, p, p, p, p, p, 1, 1, 128, 96, 0, 0.1, None) == 2
    assert lib.fa_fwd_fp8(p, p, p + 1, p, p, p, p, p, 1, 1, 128, 128, 0, 0.1, None) == 3


def test_quantiser_argument_errors_before_any_launch(lib):
    p = ALIGNED
    q = lib.fa_fp8_quantize  # (x, x_dtype, hadamard, codes, descale, rows, d, stream)
    assert q(None, 0, 0, p, p, 128, 128, None) == 1
    assert q(p, 0, 0, p, None, 128, 128, None) == 1
    assert q(p, 2, 0, p, p, 128, 128, None) == 1            # x_dtype
    assert q(p, 0, 2, p, p, 128, 128, None) == 1            # hadamard flag
    assert q(p, 0, 0, p, p, 0, 128, None) == 1              # rows
    assert q(p, 0, 0, p, p, (1 << 31) + 1, 128, None) == 1
    assert q(p, 0, 0, p, p, 128, 96, None) == 2             # d
    assert q(p + 8, 0, 0, p, p, 128, 128, None) == 3        # misaligned x

    def blk(x=p, dt=0, had=0, br=64, codes=p, desc=p, seqs=2, N=300, d=128):
        return lib.fa_fp8_quantize_blocks(x, dt, had, br, codes, desc, seqs, N, d, None)

    assert blk(br=0) == 1 and blk(br=1025) == 1
    assert blk(seqs=0) == 1 and blk(seqs=65536) == 1
    assert blk(N=0) == 1 and blk(dt=3) == 1 and blk(had=-1) == 1
    assert blk(codes=None) == 1
    assert blk(d=256) == 2
    assert blk(desc=p + 4) == 3


def test_decode_argument_errors_before_any_launch(lib):
    p = ALIGNED

    def dec(q=p, k=p, v=p, o=p, lse=p, ws=p, wsb=1 << 30, B=1, H=4, Hkv=2, N=100, d=128, scale=0.1):
        return lib.fa_decode(q, k, v, o, lse, ws, wsb, B, H, Hkv, N, d, scale, None)

    assert dec(q=None) == 1 and dec(lse=None) == 1
    assert dec(B=0) == 1 and dec(N=0) == 1
    assert dec(H=4, Hkv=3) == 1                             # Hkv must divide H
    assert dec(H=34, Hkv=2) == 1                            # groups of at most 16 query heads
    assert dec(d=96) == 2
    assert dec(scale=0.0) == 1 and dec(scale=float("inf")) == 1
    assert dec(ws=None) == 6 and dec(wsb=16) == 6           # workspace missing or too small
    assert dec(ws=p + 8) == 3
    assert dec(v=p + 4) == 3


def test_gqa_and_window_argument_errors_before_any_launch(lib):
    p = ALIGNED

    def fg(Hkv=2, causal=1, d=128):
        return lib.fa_fwd_gqa(p, p, p, p, p, 1, 4, Hkv, 128, d, causal, 0.1, None)

    def bg(Hkv=2, causal=1, ws=p, wsb=1 << 30):
        return lib.fa_bwd_gqa(p, p, p, p, p, p, p, p, p, ws, wsb, 1, 4, Hkv, 128, 128, causal, 0.1, None)

    def fw(window=16, Hkv=2):
        return lib.fa_fwd_window(p, p, p, p, p, 1, 4, Hkv, 128, 128, window, 0.1, None)

    def bw(window=16, Hkv=2, ws=p, wsb=1 << 30):
        return lib.fa_bwd_window(p, p, p, p, p, p, p, p, p, ws, wsb, 1, 4, Hkv, 128, 128, window, 0.1, None)

    assert fg(Hkv=3) == 1 and fg(Hkv=0) == 1 and fg(causal=2) == 1   # Hkv must divide H
    assert fg(d=80) == 2
    assert bg(Hkv=3) == 1 and bg(causal=5) == 1
    assert bg(ws=None) == 6 and bg(wsb=16) == 6 and bg(ws=p + 8) == 3
    assert fw(window=0) == 1 and fw(window=-5) == 1 and fw(Hkv=3) == 1
    assert bw(window=0) == 1 and bw(Hkv=3) == 1
    assert bw(ws=None) == 6 and bw(wsb=16) == 6 and bw(ws=p + 8) == 3


def test_measurement_and_exp2_hooks_reject_bad_arguments(lib):
    p = ALIGNED
    assert lib.fa_measure_ex2_rate(None, p, 1 << 20, None) == 1
    assert lib.fa_measure_ex2_rate(p, None, 1 << 20, None) == 1
    assert lib.fa_measure_ex2_rate(p, p + 4, 1 << 20, None) == 3
    assert lib.fa_debug_exp2_poly(p, p, 0, 3, None) == 1
    assert lib.fa_debug_exp2_poly(p, p, 16, 4, None) == 1
    assert lib.fa_debug_exp2_poly(None, p, 16, 3, None) == 1


def test_debug_timeout_hook_rejects_bad_limit(lib):
    assert lib.fa_debug_wait_timeout(0, None) == 1
    assert lib.fa_debug_wait_timeout(2_000_000, None) == 1


def test_product_has_no_oracle_import():
    pkg = os.path.join(ROOT, "exact_attention_76_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_build_register_check_reads_the_ptxas_report():
    log = ("ptxas info    : Compiling entry function '_ZN2fa4anon18fa_bwd_main_kernelILi128ELb0EEEv' for 'sm_103a'\n"
           "ptxas info    : Function properties for _ZN2fa4anon18fa_bwd_main_kernelILi128ELb0EEEv\n"
           "    8 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads\n"
           "ptxas info    : Used {} registers, used 2 barriers\n"
           "ptxas info    : Compiling entry function '_ZN2fa4anon18fa_bwd_main_kernelILi64ELb0EEEv' for 'sm_103a'\n"
           "ptxas info    : Used 96 registers, used 2 barriers\n")
    build.check_registers(log.format(128), "fa_bwd_main_kernelILi128E", 128, "fa_bwd.cu")
    with pytest.raises(RuntimeError, match="uses 120 registers"):
        build.check_registers(log.format(120), "fa_bwd_main_kernelILi128E", 128, "fa_bwd.cu")
    with pytest.raises(RuntimeError, match="no register report"):
        build.check_registers("", "fa_bwd_main_kernelILi128E", 128, "fa_bwd.cu")
