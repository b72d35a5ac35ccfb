"""The tcgen05 GEMM's work split (host logic, no GPU) through fs_gemm_plan,
which runs the functions fs_create and the decode step use: the properties
batch invariance and the kernels rely on, over the SmolLM2-135M and
Mistral-7B matrix shapes, handle sizes and SM counts, plus launch grids
worked out by hand from the rules."""
import itertools
import os

import pytest

from continuous_transformer_decode_gb300 import build, fs

BF16, Q8 = fs.FS_DTYPE_BF16, fs.FS_DTYPE_Q8_0

# (rows, inputs) of every weight GEMM: QKV, O, gate/up, down, LM head
SMOL = [(960, 576), (576, 576), (3072, 576), (576, 1536), (49152, 576)]
MISTRAL = [(6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336), (32000, 4096)]
HANDLES = [1, 4, 8, 16, 32, 64, 128, 256, 512, 960]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.fixture
def knobs_unset(monkeypatch):
    for k in ("FS_Q8_BF16_GROUPS",):
        monkeypatch.delenv(k, raising=False)


def _calls(max_lanes):
    return sorted({1, 2, 15, 16, 17, 31, 33, max_lanes // 2 or 1, max_lanes - 1 or 1,
                   max_lanes} & set(range(1, max_lanes + 1)))


def _cases():
    for (N, K), B, sms, dt in itertools.product(SMOL + MISTRAL, HANDLES, (152, 148, 132),
                                                (BF16, Q8)):
        yield N, K, B, sms, dt


def test_width_is_fixed_per_handle_and_splits_whole_tiles(knobs_unset):
    for N, K, B, sms, dt in _cases():
        plans = [fs.fs_gemm_plan(N, K, B, n, sms, dt) for n in _calls(B)]
        P, mt, kb = plans[0]["P"], plans[0]["m_tiles"], plans[0]["k_blocks"]
        assert mt == -(-N // 128) and kb == -(-K // 64)
        # a lane's bits may not depend on its batch: P never varies with n
        assert all(p["P"] == P for p in plans), (N, K, B, sms)
        # whole K splits of every tile, each of at least one k-block
        assert P % mt == 0 and 1 <= P // mt <= kb, (N, K, B, sms, P)
        s = P // mt
        if mt >= sms:
            assert s == 1                    # enough row tiles: whole tiles
        if B > 8:
            assert s <= 8
            if kb < 32:
                assert s == 1, (N, K, B, sms)    # short K is never split
            elif s > 1:
                assert kb // s >= (8 if B <= 32 else 32), (N, K, B, sms, s)


def test_lane_groups_cover_the_call(knobs_unset):
    for N, K, B, sms, dt in _cases():
        for n in _calls(B):
            p = fs.fs_gemm_plan(N, K, B, n, sms, dt)
            lg, g = p["lanes_per_group"], p["groups"]
            assert lg % 16 == 0 and 16 <= lg <= 128, p
            assert g == -(-n // lg) and (g - 1) * lg < n, (n, p)   # no empty group
            assert g <= 16 or g == -(-n // 128), (n, p)             # at most ~16 per tile
            t = p["tmem_cols"]
            assert t & (t - 1) == 0 and max(32, lg) <= t <= 512, p
            if dt == Q8 and not p["q8_copy_used"] and g > 1:
                assert lg >= 32, (n, p)    # Q8_0 groups each dequantise: >= 32 lanes
            if dt == BF16:
                assert p["q8_copy_kept"] == 0 and p["q8_copy_used"] == 0


def test_q8_copy_kept_and_used_where_tiles_would_be_converted_twice(monkeypatch):
    def q8_groups(N, K, B, n, sms):
        monkeypatch.setenv("FS_Q8_BF16_GROUPS", "0")    # no copies: Q8_0 grouping
        g = fs.fs_gemm_plan(N, K, B, n, sms, Q8)
        monkeypatch.delenv("FS_Q8_BF16_GROUPS")
        assert g["q8_copy_kept"] == 0 and g["q8_copy_used"] == 0
        return g["groups"]

    for (N, K), B, sms in itertools.product(SMOL + MISTRAL, HANDLES, (152, 132)):
        kept = q8_groups(N, K, B, B, sms) >= 2
        for n in _calls(B):
            p = fs.fs_gemm_plan(N, K, B, n, sms, Q8)
            assert p["q8_copy_kept"] == int(kept), (N, K, B, n)
            assert p["q8_copy_used"] == int(kept and q8_groups(N, K, B, n, sms) >= 2)
            if p["q8_copy_used"]:   # then grouped like a bf16 call
                b = fs.fs_gemm_plan(N, K, B, n, sms, BF16)
                assert (p["lanes_per_group"], p["groups"]) == (b["lanes_per_group"], b["groups"])
    # a higher threshold keeps fewer copies
    monkeypatch.setenv("FS_Q8_BF16_GROUPS", "1000")
    assert fs.fs_gemm_plan(960, 576, 960, 960, 152, Q8)["q8_copy_kept"] == 0


def _grid(N, K, B, n, sms, dt):
    p = fs.fs_gemm_plan(N, K, B, n, sms, dt)
    return p["P"] * p["groups"]


def test_launch_grids_worked_by_hand(knobs_unset):
    # SmolLM2 bf16 on a 256-lane handle, all lanes, 152 SMs. Short K, so
    # P = row tiles; fill = 2 x 152 // P blocks per tile, groups of >= 16 lanes:
    # QKV 8 tiles -> min(38, 16) = 16 groups; O and down 5 tiles -> 16;
    # gate/up 24 tiles -> 12 groups, widened to 8 groups of 32 lanes; the
    # head's 384 tiles fill the SMs alone: 256 / 128 = 2 groups
    assert [_grid(N, K, 256, 256, 152, BF16) for N, K in SMOL] == [128, 80, 192, 80, 768]
    # the same matrices at 960 Q8_0 lanes (bf16 copies): groups of >= 960 / 16
    # = 60 -> 64 lanes, 15 groups; gate/up min(12, 15) = 12; head 960 / 128
    assert [_grid(N, K, 960, 960, 152, Q8) for N, K in SMOL] == [120, 75, 288, 75, 3072]
    # Mistral-7B on a 128-lane handle: QKV 48 tiles x 2 splits (85 x 152 //
    # (100 x 48) = 2) = 96, fill 3 groups; O 32 tiles, s = min(4, 64 // 32) = 2,
    # P = 64, 4 groups; gate/up 224 tiles >= SMs: whole tiles, 1 group; down
    # 32 tiles, s = min(4, 224 // 32) = 4, P = 128, 2 groups
    assert [_grid(N, K, 128, 128, 152, BF16) for N, K in MISTRAL[:4]] == [288, 256, 224, 256]
    # a 1-lane Mistral handle: about two blocks per SM, whole splits per tile
    # (QKV 48 x min(64, 304 // 48 = 6) = 288; down 32 x 9 = 288)
    assert _grid(6144, 4096, 1, 1, 152, BF16) == 288
    assert _grid(4096, 14336, 1, 1, 152, BF16) == 288


@pytest.mark.parametrize("args", [
    (960, 570, 8, 8, 152, BF16),     # inputs not a multiple of 32
    (960, 576, 8, 9, 152, BF16),     # more lanes than the handle
    (960, 576, 8, 0, 152, BF16),
    (960, 576, 8, 8, 0, BF16),       # no SMs
    (960, 576, 8, 8, 152, fs.FS_DTYPE_F32),   # f32 weights take the GEMV
    (0, 576, 8, 8, 152, BF16),
])
def test_plan_refuses_bad_arguments(args):
    with pytest.raises(fs.FsError) as e:
        fs.fs_gemm_plan(*args)
    assert e.value.code == fs.CODES["FS_ERR_ARG"]
