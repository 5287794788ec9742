"""The C-ABI library builds, loads and exports every symbol include/fp8q.h
declares; host-only entry points (status strings, the schedule planner and
argument validation that fails before any CUDA call) work without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import fp8_w8a8_quantized_token_gb300 as fq
from fp8_w8a8_quantized_token_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fq.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^FP8Q_API\s+[\w\s\*]+?\b(fp8q_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_hot_path_entry_points():
    names = declared_functions()
    for n in ("fp8q_quant_per_token", "fp8q_quant_per_token_group_row_padded", "fp8q_scaled_mm_channelwise",
              "fp8q_scaled_mm_blockwise"):
        assert n in names
    assert set(names) == set(fq.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fq.LIB_PATH], capture_output=True, text=True, check=True)
    exported = {line.split()[-1] for line in out.stdout.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "fp8q.h"\nint main(void){ return fp8q_version() > 0 ? 0 : 1; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c", str(src),
                    "-o", str(tmp_path / "use.o")], check=True)


def test_status_strings_and_version(lib):
    assert fq.status_str(0) == "FP8Q_OK"
    assert fq.status_str(4) == "FP8Q_ERR_TIMEOUT"
    assert fq.status_str(99) == "FP8Q_UNKNOWN_STATUS"
    assert fq.fp8q_version() == (2 << 16) | 2


def test_invalid_arguments_are_rejected_before_any_cuda_call(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: validation fails first
    # K not a multiple of 16
    assert lib.fp8q_quant_per_token(fake, 4, 24, 24, fake, fake, 1e-10, None) == fq.FP8Q_ERR_INVALID_ARG
    # ldx < K
    assert lib.fp8q_quant_per_token(fake, 4, 32, 16, fake, fake, 1e-10, None) == fq.FP8Q_ERR_INVALID_ARG
    # eps <= 0
    assert lib.fp8q_quant_per_token(fake, 4, 32, 32, fake, fake, 0.0, None) == fq.FP8Q_ERR_INVALID_ARG
    # M == 0 is a no-op
    assert lib.fp8q_quant_per_token(None, 0, 32, 32, None, None, 1e-10, None) == fq.FP8Q_OK
    # group size outside {16, 32, 64, 128}
    assert lib.fp8q_quant_per_token_group_row_padded(fake, 4, 256, 256, 256, 1e-10, 4, fake, fake, 4,
                                                     None) == fq.FP8Q_ERR_UNSUPPORTED
    # m_pad not a multiple of the alignment / smaller than M
    assert lib.fp8q_quant_per_token_group_row_padded(fake, 5, 256, 256, 128, 1e-10, 4, fake, fake, 6,
                                                     None) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_quant_per_token_group_row_padded(fake, 5, 256, 256, 128, 1e-10, 4, fake, fake, 4,
                                                     None) == fq.FP8Q_ERR_INVALID_ARG
    # K not a multiple of the group
    assert lib.fp8q_quant_per_token_group_row_padded(fake, 4, 192, 192, 128, 1e-10, 4, fake, fake, 4,
                                                     None) == fq.FP8Q_ERR_INVALID_ARG
    # blockwise needs N, K multiples of 128 (the reference falls back; we refuse)
    assert lib.fp8q_scaled_mm_blockwise(fake, fake, fake, fake, None, fake, 4, 4, 200, 256, 0, None, 0,
                                        None) == fq.FP8Q_ERR_UNSUPPORTED
    assert lib.fp8q_scaled_mm_blockwise(fake, fake, fake, fake, None, fake, 4, 4, 256, 200, 0, None, 0,
                                        None) == fq.FP8Q_ERR_UNSUPPORTED
    assert lib.fp8q_scaled_mm_blockwise(fake, fake, fake, fake, None, fake, 5, 6, 256, 256, 0, None, 0,
                                        None) == fq.FP8Q_ERR_INVALID_ARG
    # channelwise: K % 16, ldb < K, N % 8, unknown output type, misaligned pointer
    assert lib.fp8q_scaled_mm_channelwise(fake, fake, 40, fake, fake, None, fake, 4, 64, 40, 0, None, 0,
                                          None) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_scaled_mm_channelwise(fake, fake, 32, fake, fake, None, fake, 4, 64, 64, 0, None, 0,
                                          None) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_scaled_mm_channelwise(fake, fake, 64, fake, fake, None, fake, 4, 60, 64, 0, None, 0,
                                          None) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_scaled_mm_channelwise(fake, fake, 64, fake, fake, None, fake, 4, 64, 64, 7, None, 0,
                                          None) == fq.FP8Q_ERR_UNSUPPORTED
    assert lib.fp8q_scaled_mm_channelwise(P(0x1008), fake, 64, fake, fake, None, fake, 4, 64, 64, 0, None, 0,
                                          None) == fq.FP8Q_ERR_INVALID_ARG
    # null pointers
    assert lib.fp8q_scaled_mm_channelwise(None, fake, 64, fake, fake, None, fake, 4, 64, 64, 0, None, 0,
                                          None) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_scaled_mm_channelwise(None, None, 64, None, None, None, None, 0, 64, 64, 0, None, 0,
                                          None) == fq.FP8Q_OK
    # a workspace that is not 16-byte aligned
    assert lib.fp8q_scaled_mm_channelwise(fake, fake, 64, fake, fake, None, fake, 4, 64, 64, 0, P(0x1004), 4096,
                                          None) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_scaled_mm_blockwise(fake, fake, fake, fake, None, fake, 4, 4, 256, 256, 0, P(0x1008), 4096,
                                        None) == fq.FP8Q_ERR_INVALID_ARG
    # invalid sizes need no workspace
    for M, N, K in ((0, 64, 64), (-1, 64, 64), (4, 0, 64), (4, 64, 0)):
        assert lib.fp8q_workspace_bytes(M, N, K, 0) == 0


def test_plan_override_validation(lib):
    assert lib.fp8q_set_plan_override(1, 48, 1) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_set_plan_override(0, 16, 1) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_set_plan_override(1, 32, -1) == fq.FP8Q_ERR_INVALID_ARG
    assert lib.fp8q_set_plan_override(0, 256, 0) == fq.FP8Q_ERR_INVALID_ARG   # stream-K: swapped tiles only
    assert lib.fp8q_set_plan_override(1, 32, 0) == fq.FP8Q_OK
    p = fq.fp8q_gemm_plan(7, 4096, 4096, num_sms=148)
    assert (p["swap_ab"], p["mma_n"], p["split_k"], p["stream_k"]) == (1, 32, 1, 1)
    assert lib.fp8q_set_plan_override(1, 32, 3) == fq.FP8Q_OK
    p = fq.fp8q_gemm_plan(7, 4096, 4096, num_sms=148)
    assert (p["swap_ab"], p["mma_n"], p["split_k"], p["from_table"]) == (1, 32, 3, 0)
    assert lib.fp8q_set_plan_override(-1, 0, 0) == fq.FP8Q_OK


def test_variant_entry_points_reject_invalid_arguments_before_any_cuda_call(lib):
    """The variant, linear and weight-only entry points validate every
    argument first: each case below fails (or, M = 0, succeeds as a no-op)
    without touching the device, so it runs without a GPU."""
    P = ctypes.c_void_p
    fake, odd = P(0x1000), P(0x1001)   # never dereferenced
    E = fq.FP8Q_ERR_INVALID_ARG
    U = fq.FP8Q_ERR_UNSUPPORTED
    g = lib.fp8q_quant_per_token_group_row_padded_ex
    assert g(fake, 4, 256, 256, 128, 1e-10, 4, 8, fake, fake, 4, None) == E          # unknown flag bit
    assert g(fake, 4, 256, 256, 48, 1e-10, 4, 0, fake, fake, 4, None) == U           # group size 48
    assert g(fake, 4, 256, 256, 0, 1e-10, 4, 0, fake, fake, 4, None) == E            # group size 0
    assert g(fake, 4, 256, 256, 128, 1e-10, 4, 2, fake, fake, 4, None) == E          # silu: ldx < 2K
    assert g(fake, 5, 256, 256, 128, 1e-10, 4, 1, fake, fake, 6, None) == E          # m_pad % alignment
    assert g(None, 0, 256, 512, 64, 1e-10, 4, 3, None, None, 0, None) == fq.FP8Q_OK  # M = 0
    s = lib.fp8q_quant_static_per_tensor
    assert s(fake, 4, 24, 24, fake, fake, None, None) == E                           # K % 16
    assert s(fake, 4, 32, 16, fake, fake, None, None) == E                           # ldx < K
    assert s(fake, 4, 32, 32, None, fake, None, None) == E                           # no scale
    assert s(P(0x1008), 4, 32, 32, fake, fake, None, None) == E                      # x not 16-byte aligned
    assert s(None, 0, 32, 32, None, None, None, None) == fq.FP8Q_OK                  # M = 0
    wb = lib.fp8q_quant_weight_block128
    assert wb(fake, 200, 256, fake, fake, 1e-10, None) == U                          # N % 128
    assert wb(fake, 256, 256, fake, fake, 0.0, None) == E                            # eps
    lc = lib.fp8q_linear_channelwise
    assert lc(fake, fake, 64, fake, None, fake, 4, 64, 64, fake, fake, 7, None, 0, None) == U  # output type
    assert lc(fake, fake, 64, fake, None, fake, 4, 60, 64, fake, fake, 0, None, 0, None) == E  # N % 8
    assert lc(None, None, 64, None, None, None, 0, 64, 64, None, None, 0, None, 0, None) == fq.FP8Q_OK
    lb = lib.fp8q_linear_blockwise
    assert lb(fake, fake, fake, None, fake, 4, 200, 256, fake, fake, 4, 0, None, 0, None) == U  # N % 128
    assert lb(fake, fake, fake, None, fake, 5, 256, 256, fake, fake, 6, 0, None, 0, None) == E  # m_pad % 4
    assert lb(fake, fake, fake, odd, fake, 4, 256, 256, fake, fake, 4, 0, None, 0, None) == E   # odd bias address
    fu = lib.fp8q_linear_blockwise_fused
    assert fu(fake, 256, fake, fake, None, fake, 4, 200, 256, 0, None) == U           # N % 128
    assert fu(fake, 128, fake, fake, None, fake, 4, 256, 256, 0, None) == E           # ldx < K
    assert fu(fake, 256, fake, fake, odd, fake, 4, 256, 256, 0, None) == E            # odd bias address
    assert fu(None, 256, None, None, None, None, 0, 256, 256, 0, None) == fq.FP8Q_OK  # M = 0
    w16 = lib.fp8q_scaled_mm_w8a16
    assert w16(fake, 40, fake, 48, fake, None, fake, 4, 64, 40, 0, None) == E         # K % 16
    assert w16(fake, 64, fake, 72, fake, None, fake, 4, 64, 64, 0, None) == E         # ldw % 16
    assert w16(fake, 64, fake, 64, fake, None, fake, 4, 60, 64, 0, None) == E         # N % 8
    assert w16(fake, 64, fake, 64, fake, None, fake, 4, 64, 64, 5, None) == U         # output type
    assert w16(fake, 64, None, 64, fake, None, fake, 4, 64, 64, 0, None) == E         # no weights
    assert w16(fake, 64, fake, 64, fake, odd, fake, 4, 64, 64, 0, None) == E          # odd bias address
    assert w16(None, 64, None, 64, None, None, None, 0, 64, 64, 0, None) == fq.FP8Q_OK
    na = lib.fp8q_linear_channelwise_noalloc
    assert na(fake, fake, 64, fake, None, fake, 4, 64, 0, 0, None) == E               # K <= 0
    assert na(None, None, 64, None, None, None, 0, 64, 64, 0, None) == fq.FP8Q_OK     # M = 0
