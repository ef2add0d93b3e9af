"""Host-side model of the verify kernel's cost-balanced partition (no GPU).

The split kernel's CTAs cut equal shares of a cost that counts every
(lane, kv head) unit as its pages plus a unit cost (the price of starting a
unit, in pages of the cache format: 20 for FP8 page scales, 16 for the
others), map
their cost interval back to page positions, and the
merge finds a unit's first and last CTA from cost positions.  This model
states those rules in Python and checks the invariants the kernel relies on
at sizes the GPU tests do not reach: the CTAs' page ranges tile every page
exactly once, the merge's CTA range is exactly the CTAs that hold a unit's
pages, and the kernel's 32-bit floor(c * T / Ce) and fp32-estimated inverse
agree with exact arithmetic for every total cost below 2^31."""
import numpy as np
import pytest

UNIT_COSTS = (16, 20)  # FP8 row, INT4, INT8; FP8 page scales


def prefix(pages, UNIT_COST):
    pref, cp = [0], [0]
    for n in pages:
        pref.append(pref[-1] + n)
        cp.append(cp[-1] + (n + UNIT_COST if n > 0 else 0))
    return pref, cp


def real_of(y, pref, cp, H, UNIT_COST):
    B = len(pref) - 1
    if y >= H * cp[B]:
        return H * pref[B]
    lo = max(b for b in range(B) if H * cp[b] <= y)
    nb = pref[lo + 1] - pref[lo]
    r = y - H * cp[lo]
    q, v = divmod(r, nb + UNIT_COST)
    return H * pref[lo] + q * nb + max(0, v - UNIT_COST)


def cost_begin_u32(c, ce, T):
    """The kernel's floor(c T / Ce) in unsigned 32-bit arithmetic."""
    u = np.uint32
    T, ce, cc = u(T), u(ce), u(c)
    with np.errstate(over="raise"):
        qT = T // ce
        rT = T - qT * ce
        return int(cc * qT + (cc * rT) // ce)


def cta_of_cost(y, ce, T):
    """The kernel's inverse: an fp32 estimate, then exact steps."""
    c = int(np.float32(y) * np.float32(ce) / np.float32(T))
    c = max(0, min(c, ce - 1))
    while c > 0 and cost_begin_u32(c, ce, T) > y:
        c -= 1
    while c + 1 < ce and cost_begin_u32(c + 1, ce, T) <= y:
        c += 1
    return c


def check(pages, H, C, UNIT_COST):
    pref, cp = prefix(pages, UNIT_COST)
    T, P = H * cp[-1], H * pref[-1]
    if T == 0:
        return
    ce = min(C, T)
    begins = [real_of(cost_begin_u32(c, ce, T), pref, cp, H, UNIT_COST) for c in range(ce + 1)]
    assert begins[0] == 0 and begins[-1] == P
    assert all(begins[i] <= begins[i + 1] for i in range(ce))
    for b, nb in enumerate(pages):
        if nb == 0:
            continue
        for hk in range(H):
            first_page = H * pref[b] + hk * nb
            y0 = H * cp[b] + hk * (nb + UNIT_COST) + UNIT_COST  # cost position of the unit's first page
            f, l = cta_of_cost(y0, ce, T), cta_of_cost(y0 + nb - 1, ce, T)
            for c in range(ce):
                holds = max(begins[c], first_page) < min(begins[c + 1], first_page + nb)
                assert holds == (f <= c <= l), (pages, H, C, b, hk, c, f, l)


@pytest.mark.parametrize("unit_cost", UNIT_COSTS)
def test_random_lane_mixes_tile_and_invert(unit_cost):
    rng = np.random.default_rng(5)
    for _ in range(600):
        B = int(rng.integers(1, 40))
        pages = [int(rng.choice([0, 1, 2, rng.integers(1, 50), rng.integers(1, 2000)])) for _ in range(B)]
        check(pages, int(rng.choice([1, 2, 4, 8])), int(rng.choice([1, 3, 148, 152, 1024])), unit_cost)


@pytest.mark.parametrize("unit_cost", UNIT_COSTS)
def test_workload_shapes(unit_cost):
    check([114, 290, 394, 487, 491, 864, 978, 1011], 4, 148, unit_cost)  # eight lanes of 4k..64k tokens
    check([3751], 4, 148, unit_cost)                                       # one lane of 240,000 tokens
    check([512], 4, 148, unit_cost)                                        # plain decode of 32,768 tokens


@pytest.mark.parametrize("T", [1, 7, 1023, 1024, 2**20 + 3, 2**31 - 1, 2**31 - 1025, 1_500_000_017])
def test_32bit_floor_and_inverse_up_to_2_31(T):
    rng = np.random.default_rng(T % 1000)
    for ce in sorted({1, 2, 148, 152, 1024, min(T, 1000), min(T, 1024)}):
        if ce > T:
            continue
        for c in list(range(0, min(ce, 40) + 1)) + [int(x) for x in rng.integers(0, ce + 1, size=40)] + [ce]:
            assert cost_begin_u32(c, ce, T) == (c * T) // ce, (c, ce, T)
        for y in [0, T - 1] + [int(x) for x in rng.integers(0, T, size=60)]:
            c = cta_of_cost(y, ce, T)
            assert (c * T) // ce <= y < ((c + 1) * T) // ce or (c == ce - 1 and y >= (c * T) // ce), (y, ce, T, c)
