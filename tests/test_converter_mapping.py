"""The split kernel's converter index mapping, restated and checked on CPU.

Converter thread u (kCT threads: 128 with four converter warps, 256 with
eight) handles the items u, u + kCT, ... of a page.  Lane l of a warp takes
a row offset and a chunk (FP8, INT8: 16-dim chunk c of a 128-byte row) or a
group (INT4: 32-dim group of a 64-byte row) so that each quarter-warp (8
lanes, the unit in which shared memory serves 16-byte accesses) spans two
key rows.  These tests check that every item of a page is covered exactly
once, and that each quarter-warp's 16-byte loads (the codes) and stores (the
fp16 tile, 16-byte chunk k of row r at r * 128 + ((k ^ (r & 7)) << 4), the
two 8 KB dim halves sharing banks) fall in 8 distinct 16-byte bank groups."""
import pytest


def lane_terms(lane):
    q8, rr = lane >> 3, (lane >> 2) & 1
    c8 = (lane & 3) + 4 * (rr ^ (q8 & 1))
    rof8 = 2 * (q8 >> 1) + rr
    hb, r4 = (lane >> 2) & 1, (lane >> 1) & 1
    g4 = (lane & 1) + 2 * (hb ^ (q8 & 1))
    rof4 = 4 * (q8 >> 1) + 2 * hb + r4
    return c8, rof8, g4, rof4


def fp8_item(item):  # FP8 formats: V only, 512 chunks (64 rows x 8)
    c8, rof8, _, _ = lane_terms(item & 31)
    return 0, 4 * (item >> 5) + rof8, c8


def int8_item(item):  # INT8: K and V, 1024 chunks
    c8, rof8, _, _ = lane_terms(item & 31)
    return item >> 9, 4 * ((item & 511) >> 5) + rof8, c8


def int4_item(item):  # INT4: K and V, 512 groups (64 rows x 4 per tile)
    _, _, g4, rof4 = lane_terms(item & 31)
    return item >> 8, 8 * ((item & 255) >> 5) + rof4, g4


def c8_load_bank(fmt, tk, r, c):
    # FP8: the TMA tile with the 128-byte swizzle; INT8: plain 128-byte code rows
    return (c ^ (r & 7)) if fmt == "fp8" else c


def c8_store_banks(tk, r, c):
    c0 = 2 * (c & 3)
    return [(c0 ^ (r & 7)), ((c0 + 1) ^ (r & 7))]


def i4_load_bank(tk, r, gi):
    return (r * 64 + gi * 16) // 16 % 8


def i4_store_banks(tk, r, gi):
    return [((4 * (gi & 1) + k) ^ (r & 7)) for k in range(4)]


CASES = [("fp8", fp8_item, 512), ("int8", int8_item, 1024), ("int4", int4_item, 512)]


# (format, converter threads): FP8 formats and INT4 run four converter warps, INT8 eight;
# the mapping is also checked for the other count of the INT formats
ONCE = [(c[0], c[1], c[2], kct) for c in CASES for kct in ((128,) if c[0] == "fp8" else (128, 256))]


@pytest.mark.parametrize("fmt,item_of,n,kct", ONCE, ids=[f"{c[0]}-{c[3]}" for c in ONCE])
def test_every_item_once(fmt, item_of, n, kct):
    seen = {}
    for u in range(kct):
        for q in range(n // kct):
            key = item_of(u + kct * q)
            assert key not in seen, (fmt, kct, u, q, key)
            seen[key] = (u, q)
    rows = 64
    per_row = 8 if fmt != "int4" else 4
    tiles = 1 if fmt == "fp8" else 2
    assert len(seen) == n == tiles * rows * per_row
    assert all(0 <= r < rows for (_, r, _) in seen)


@pytest.mark.parametrize("fmt,item_of,n", CASES, ids=[c[0] for c in CASES])
def test_quarter_warps_are_conflict_free(fmt, item_of, n):
    for w0 in range(0, n, 32):
        for q0 in range(w0, w0 + 32, 8):
            ids = [item_of(i) for i in range(q0, q0 + 8)]
            if fmt == "int4":
                loads = [i4_load_bank(*x) for x in ids]
                stores = [i4_store_banks(*x) for x in ids]
            else:
                loads = [c8_load_bank(fmt, *x) for x in ids]
                stores = [c8_store_banks(*x) for x in ids]
            assert len(set(loads)) == 8, (fmt, q0, loads)
            for k in range(len(stores[0])):
                assert len({s[k] for s in stores}) == 8, (fmt, q0, k)


def test_the_previous_mapping_had_two_way_conflicts():
    # one row per quarter-warp (chunks c and c + 4 share banks in the fp16 tile)
    ids = [(0, 0, c) for c in range(8)]
    assert len({c8_store_banks(*x)[0] for x in ids}) == 4
