"""Host-side schedule selection (no GPU needed): every plan the library can
produce launches a kernel instantiation that exists, covers every tile once,
splits K only across whole 128-wide K blocks and stays inside the shared
memory budget."""
import itertools

import pytest

import fp8_w8a8_quantized_token_gb300 as fq
from fp8_w8a8_quantized_token_gb300 import build as fbuild

SUPPORTED = {(1, 16), (1, 32), (1, 64), (1, 128), (0, 32), (0, 64), (0, 128), (0, 256)}
SMEM_LIMIT = 232448


@pytest.fixture(scope="module", autouse=True)
def lib():
    fbuild.build()
    L = fq.load_library()
    L.fp8q_set_plan_override(-1, 0, 0)
    return L


def stage_bytes(swap, mma_n, blockwise):
    tok_tile = mma_n if swap else 128
    return 128 * 128 + mma_n * 128 + (tok_tile * 4 if blockwise else 0)


SHAPES = [(4096, 4096), (6144, 4096), (4096, 12288), (24576, 4096), (4096, 7168), (24576, 3072), (3072, 12288),
          (256, 512), (384, 1040)]
MS = [1, 2, 3, 4, 5, 7, 13, 16, 31, 32, 64, 100, 128, 129, 256, 512, 1024, 2048, 4096, 8192]


@pytest.mark.parametrize("num_sms", [148, 152])
def test_plans_are_launchable(num_sms):
    for (N, K), M, bw in itertools.product(SHAPES, MS, (0, 1)):
        if bw and (N % 128 or K % 128):
            continue
        p = fq.fp8q_gemm_plan(M, N, K, bool(bw), num_sms=num_sms)
        assert (p["swap_ab"], p["mma_n"]) in SUPPORTED
        assert p["tile_m"] == (p["mma_n"] if p["swap_ab"] else 128)
        assert p["tile_n"] == (128 if p["swap_ab"] else p["mma_n"])
        tiles = -(-M // p["tile_m"]) * -(-N // p["tile_n"])
        num_kb = -(-K // 128)
        assert 1 <= p["split_k"] <= min(8, num_kb)
        if p["stream_k"]:
            # stream-K: swapped tiles, no clusters, one CTA per SM at most and
            # at least one (tile, K block) pair per CTA
            assert p["swap_ab"] == 1 and p["split_k"] == 1 and p["pair"] == 0 and p["persistent"] == 1
            assert p["grid"] == min(tiles * num_kb, num_sms)
            assert p["kb_per_stage"] == 1
            assert p["stages"] * stage_bytes(1, p["mma_n"], bw) + 4096 <= SMEM_LIMIT
            continue
        m_tiles = -(-M // p["tile_m"])
        # channelwise 256-column tiles pair up (blockwise and narrower tiles never do)
        assert p["pair"] == int(not bw and not p["swap_ab"] and p["mma_n"] == 256 and p["split_k"] == 1
                                and m_tiles >= 2)
        if p["pair"]:
            # 2-CTA clusters over pairs of token tiles (an odd last tile pairs
            # with an empty one), at most one pair per two SMs
            pairs = -(-m_tiles // 2) * -(-N // p["tile_n"])
            assert p["grid"] == 2 * min(pairs, num_sms // 2)
            assert p["persistent"] == int(pairs > num_sms // 2)
        elif p["split_k"] > 1:
            assert p["grid"] == tiles * p["split_k"] and not p["persistent"]
        else:
            assert p["grid"] == min(tiles, num_sms)
            assert p["persistent"] == int(tiles > num_sms)
        # channelwise pairs of 128 x 256 tiles use 2-CTA MMAs: each CTA stages
        # 128 token rows and its 128 of the 256 weight rows per K slice
        assert p["two_sm"] == p["pair"]
        # narrow channelwise tiles over whole K blocks, K not split: two K
        # blocks per stage
        wide = (not bw and not p["swap_ab"] and not p["pair"] and p["split_k"] == 1 and K % 128 == 0
                and p["mma_n"] <= 128)
        assert p["kb_per_stage"] == (2 if wide else 1)
        per_stage = 2 * 128 * 128 if p["two_sm"] else stage_bytes(p["swap_ab"], p["mma_n"], bw)
        assert p["stages"] * per_stage * p["kb_per_stage"] + 4096 <= SMEM_LIMIT


def test_decode_sizes_put_weights_on_the_mma_m_side():
    for M in (1, 8, 16, 33, 64):
        for N, K in ((4096, 4096), (8000, 1024)):   # a tabulated and an untabulated shape
            assert fq.fp8q_gemm_plan(M, N, K, num_sms=148)["swap_ab"] == 1


def test_override_forces_the_schedule_and_clamps_split():
    try:
        fq.fp8q_set_plan_override(0, 256, 16)
        p = fq.fp8q_gemm_plan(300, 4096, 512, num_sms=148)
        assert (p["swap_ab"], p["mma_n"], p["split_k"]) == (0, 256, 4)   # 512 / 128 = 4 K blocks
        fq.fp8q_set_plan_override(1, 16, 20)
        assert fq.fp8q_gemm_plan(1, 4096, 4096, num_sms=148)["split_k"] == 8
    finally:
        fq.fp8q_set_plan_override(-1)


@pytest.mark.parametrize("num_sms", [148, 152])
def test_stream_k_plans(num_sms):
    """split_k 0 on swapped tiles asks for stream-K: split 1, no pairs, one
    CTA per SM at most, at least one (tile, K block) pair per CTA."""
    try:
        fq.fp8q_set_plan_override(1, 16, 0)
        p = fq.fp8q_gemm_plan(16, 24576, 4096, num_sms=num_sms)      # 192 tiles x 32 K blocks
        assert (p["stream_k"], p["split_k"], p["pair"], p["grid"], p["persistent"]) == (1, 1, 0, num_sms, 1)
        p = fq.fp8q_gemm_plan(1, 256, 512, num_sms=num_sms)          # 2 tiles x 4 K blocks = 8 pairs
        assert (p["stream_k"], p["grid"]) == (1, 8)
        fq.fp8q_set_plan_override(1, 32, 0)
        p = fq.fp8q_gemm_plan(32, 4096, 12288, blockwise=True, num_sms=num_sms)
        assert p["stream_k"] == 1 and p["mma_n"] == 32 and p["tile_m"] == 32
        assert fq.load_library().fp8q_set_plan_override(1, 64, 0) == fq.FP8Q_ERR_INVALID_ARG
        fq.fp8q_set_plan_override(1, 16, 4)
        assert fq.fp8q_gemm_plan(16, 24576, 4096, num_sms=num_sms)["stream_k"] == 0
    finally:
        fq.fp8q_set_plan_override(-1)


def load_table():
    import os
    import re
    path = os.path.join(os.path.dirname(fq.__file__), "csrc", "tile_table.inc")
    rows = []
    for line in open(path):
        m = re.match(r"\s*\{(-?\d+), (-?\d+), (-?\d+), (-?\d+), (-?\d+), (-?\d+), (-?\d+)\},", line)
        if m:
            rows.append(tuple(int(v) for v in m.groups()))
    return rows


def test_table_lookup_is_nearest_m_with_ties_to_the_smaller_m():
    """The rule of get_w8a8_channelwise_fp8_config: the entry of the key
    nearest to M, keys scanned in ascending order, so a tie goes to the
    smaller key -- among the keys whose schedule M does not push to more
    token tiles than the key itself had (while a key >= M exists)."""
    rows = load_table()
    assert rows, "the sweep table is empty"
    by_shape = {}
    for N, K, bw, M, swap, mma_n, split in rows:
        by_shape.setdefault((N, K, bw), []).append((M, (swap, mma_n, split)))
    for (N, K, bw), entries in by_shape.items():
        entries.sort()
        keys = [m for m, _ in entries]
        table = dict(entries)
        probe = sorted(set(keys + [(a + b) // 2 for a, b in zip(keys, keys[1:])] + [k + 1 for k in keys] + [3, 10000]))
        def tiles(k, m):
            swap, mma_n, _ = table[k]
            tm = mma_n if swap else 128
            return -(-m // tm)
        for M in probe:
            ok = [k for k in keys if not (k < M and max(keys) >= M and tiles(k, M) > tiles(k, k))]
            best = min(ok, key=lambda k: abs(k - M))   # Python's min keeps the first (smallest) on ties
            swap, mma_n, split = table[best]
            p = fq.fp8q_gemm_plan(M, N, K, bool(bw), num_sms=148)
            assert p["from_table"] == 1
            assert (p["swap_ab"], p["mma_n"]) == (swap, mma_n), (N, K, bw, M, best)
            if split == 0:   # stream-K row
                assert p["stream_k"] == 1 and p["split_k"] == 1, (N, K, bw, M, best)
            else:
                assert p["stream_k"] == 0
                assert p["split_k"] == min(split, 8, -(-K // 128)), (N, K, bw, M, best)


def test_shapes_without_rows_use_the_generic_rule():
    p = fq.fp8q_gemm_plan(7, 1000 * 8, 1024, num_sms=148)
    assert p["from_table"] == 0 and p["swap_ab"] == 1 and p["mma_n"] == 16
    assert p["split_k"] in (1, 2, 4, 8)
    p = fq.fp8q_gemm_plan(4000, 8000, 1024, num_sms=148)
    assert p["from_table"] == 0 and (p["swap_ab"], p["mma_n"], p["split_k"]) == (0, 256, 1)


def test_tuner_only_proposes_schedules_the_library_accepts(lib):
    """tune.py's candidate schedules for every swept (shape, M) are ones the
    plan override accepts and that fp8q_gemm_plan then launches as a
    supported instantiation; the non-swapped 256 tile is always among them."""
    from fp8_w8a8_quantized_token_gb300 import tune
    try:
        for label, (N, K, bw, ms) in tune.SHAPES.items():
            for M in ms:
                cands = tune.candidates(M)
                assert any(c[:2] == (0, 256) for c in cands), (label, M)
                for c in cands:
                    assert (c[0], c[1]) in SUPPORTED, (label, M, c)
                    assert c[2] in (tune.SWAP_SPLITS if c[0] else tune.SPLITS), (label, M, c)
                    assert lib.fp8q_set_plan_override(*c) == fq.FP8Q_OK
                    plan = fq.fp8q_gemm_plan(M, N, K, bool(bw), num_sms=152)
                    assert (plan["swap_ab"], plan["mma_n"]) == (c[0], c[1]), (label, M, c, plan)
    finally:
        lib.fp8q_set_plan_override(-1, 0, 0)


def test_linear_channelwise_launch_count(lib):
    """One token with rows up to 12288 values (channelwise: on layers of at
    most 4096 x 4096 weights): one fused launch; otherwise the quantizer and
    the GEMM; nothing for empty problems; two again while a schedule override
    asks for the GEMM."""
    assert fq.fp8q_linear_channelwise_launches(1, 4096, 4096) == 1
    assert fq.fp8q_linear_channelwise_launches(1, 8, 16) == 1
    assert fq.fp8q_linear_channelwise_launches(1, 136, 4112) == 1
    assert fq.fp8q_linear_channelwise_launches(1, 136, 12288) == 1
    assert fq.fp8q_linear_channelwise_launches(1, 136, 12304) == 2
    assert fq.fp8q_linear_channelwise_launches(1, 6144, 4096) == 2     # larger layers: two kernels
    assert fq.fp8q_linear_channelwise_launches(1, 4096, 12288) == 2
    assert fq.fp8q_linear_channelwise_launches(1, 24576, 4096) == 2
    assert fq.fp8q_linear_channelwise_launches(2, 4096, 4096) == 2
    assert fq.fp8q_linear_channelwise_launches(8192, 4096, 4096) == 2
    assert fq.fp8q_linear_channelwise_launches(0, 4096, 4096) == 0
    assert fq.fp8q_linear_blockwise_launches(1, 7168) == 1
    assert fq.fp8q_linear_blockwise_launches(1, 12288) == 1
    assert fq.fp8q_linear_blockwise_launches(1, 12416) == 2
    assert fq.fp8q_linear_blockwise_launches(2, 7168) == 2
    assert fq.fp8q_linear_blockwise_launches(0, 7168) == 0
    lib.fp8q_set_plan_override(1, 16, 4)
    try:
        assert fq.fp8q_linear_channelwise_launches(1, 4096, 4096) == 2
        assert fq.fp8q_linear_blockwise_launches(1, 7168) == 2
    finally:
        lib.fp8q_set_plan_override(-1, 0, 0)
