"""The bank-row layout, checked on the CPU.

moe_pack_expert runs the same host-side packing as moe_init_banks.  Each test
packs random experts and decodes the row with a decoder written from the
layout's description in include/moe_residency.h (independent of the packing
code); the decode must reproduce every logical code and scale byte."""
import numpy as np
import pytest

import cold_expert_residency_gb300 as moe

GROUP = 8704          # 128 rows x 64 code bytes + a 512-byte scale atom


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.lib()


def random_expert(rng, H, I):
    w13_q = rng.integers(0, 256, size=(2 * I, H // 2), dtype=np.uint8)
    w13_s = rng.integers(104, 141, size=(2 * I, H // 32), dtype=np.uint8)
    w2_q = rng.integers(0, 256, size=(H, I // 2), dtype=np.uint8)
    w2_s = rng.integers(104, 141, size=(H, I // 32), dtype=np.uint8)
    return w13_q, w13_s, w2_q, w2_s


def put_block(blk, q, s, rows, kblocks, box_kb):
    """Copy one 8704-byte block's codes and scales into the logical arrays:
    tile row m -> logical row rows[m]; the block's K blocks box_kb[i] hold the
    row's 32-element blocks kblocks[i]."""
    codes = blk[:8192].reshape(128, 64)
    atom = blk[8192:]
    m = np.arange(128)
    for kb, lb in zip(box_kb, kblocks):
        q[rows, lb * 16:(lb + 1) * 16] = codes[:, kb * 16:(kb + 1) * 16]
        s[rows, lb] = atom[(m % 32) * 16 + 4 * (m // 32) + kb]


def decode_row(row, H, I):
    w13_q = np.zeros((2 * I, H // 2), np.uint8)
    w13_s = np.zeros((2 * I, H // 32), np.uint8)
    w2_q = np.zeros((H, I // 2), np.uint8)
    w2_s = np.zeros((H, I // 32), np.uint8)
    m = np.arange(128)
    w, l = m // 32, m % 32
    g13 = H // 128
    for mt in range(I // 64):
        rows = np.where(l < 16, 0, I) + 64 * mt + 16 * w + l % 16
        for s in range(g13):
            off = (mt * g13 + s) * GROUP
            put_block(row[off:off + GROUP], w13_q, w13_s, rows, [4 * s + i for i in range(4)], range(4))
    base = (I // 64) * g13 * GROUP
    gfull, half = I // 128, (I // 64) % 2
    for mt in range(H // 128):
        rows = 128 * mt + m
        if not half:
            for s in range(gfull):
                off = base + (mt * gfull + s) * GROUP
                put_block(row[off:off + GROUP], w2_q, w2_s, rows, [4 * s + i for i in range(4)], range(4))
        else:
            pair = base + (mt // 2) * (2 * gfull + 1) * GROUP
            for s in range(gfull):
                off = pair + ((mt % 2) * gfull + s) * GROUP
                put_block(row[off:off + GROUP], w2_q, w2_s, rows, [4 * s + i for i in range(4)], range(4))
            off = pair + 2 * gfull * GROUP
            kb0 = 2 * (mt % 2)
            put_block(row[off:off + GROUP], w2_q, w2_s, rows, [4 * gfull, 4 * gfull + 1], [kb0, kb0 + 1])
    return w13_q, w13_s, w2_q, w2_s


@pytest.mark.parametrize("H,I", [(256, 128), (256, 192), (512, 64), (384, 128), (512, 320)])
def test_packed_row_decodes_to_the_logical_expert(lib, H, I):
    rng = np.random.default_rng(H * 1000 + I)
    expert = random_expert(rng, H, I)
    row = moe.moe_pack_expert(H, I, *expert)
    assert row.size == moe.moe_expert_bytes(H, I)
    for got, want, name in zip(decode_row(row, H, I), expert, ("w13_q", "w13_s", "w2_q", "w2_s")):
        assert np.array_equal(got, want), name


def test_row_is_a_permutation_of_the_logical_bytes(lib):
    # every logical byte lands exactly once: the row holds exactly the
    # expert's bytes, no padding
    H, I = 256, 192
    rng = np.random.default_rng(7)
    expert = random_expert(rng, H, I)
    row = moe.moe_pack_expert(H, I, *expert)
    logical = np.concatenate([a.ravel() for a in expert])
    assert row.size == logical.size
    assert np.array_equal(np.bincount(row, minlength=256), np.bincount(logical, minlength=256))


def test_pack_rejects_bad_geometry_and_scales(lib):
    rng = np.random.default_rng(1)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_pack_expert(384, 192, *random_expert(rng, 384, 192))   # odd W2 tile count with a half group
    assert ei.value.code == moe.MOE_EINVAL
    w13_q, w13_s, w2_q, w2_s = random_expert(rng, 256, 128)
    w2_s[3, 1] = 141
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_pack_expert(256, 128, w13_q, w13_s, w2_q, w2_s)
    assert ei.value.code == moe.MOE_EINVAL
