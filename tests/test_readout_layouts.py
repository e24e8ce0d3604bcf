"""Index arithmetic of the two coalesced TMEM read-outs, checked on the CPU (no GPU).

* tmem_rows_to_global_xpose (csrc/fa_ptx.cuh, used by the dK/dV pass): lane l of a warp holds
  the U = NCOLS/8 16-byte units of row l; a butterfly of xor shuffles (stage s = U/2 .. 1: for
  each unit pair (e, e|s) with bit s clear in e, the lane with bit s set sends unit e and keeps
  the received one there, the other lane sends unit e|s) must leave lane g*U + i holding unit i
  of rows g*U + e in slot e, so that store e writes U contiguous units of one row per group.
* tmem_rows_to_global_staged (csrc/fa_ptx.cuh, used by both forwards): row r of a warp's 4 KB
  buffer at 128 r, 16-byte unit u at ((u ^ (r % 8)) * 16).  Lane = row writes unit u (for each
  u); in the read-back store k lane l reads unit l % 8 of row 4k + l / 8.  Both access patterns
  must be free of shared-memory bank conflicts (a 16-byte-per-lane access is served in four
  phases of 8 lanes; 8 lanes with 8 distinct 16-byte bank groups are conflict-free), and the
  read-back must cover every unit of every row exactly once.
Planted mistakes (a wrong shuffle partner, a missing XOR) must be caught.
"""
import pytest


def butterfly(U, partner=lambda l, s: l ^ s):
    m = [[(lane, u) for u in range(U)] for lane in range(32)]  # (row, unit) each slot holds
    s = U // 2
    while s >= 1:
        for e in range(U):
            if e & s:
                continue
            send = [m[l][e] if (l & s) else m[l][e | s] for l in range(32)]
            recv = [send[partner(l, s)] for l in range(32)]
            for l in range(32):
                if l & s:
                    m[l][e] = recv[l]
                else:
                    m[l][e | s] = recv[l]
        s //= 2
    return m


def xpose_ok(U, m):
    for l in range(32):
        g, i = divmod(l, U)
        for e in range(U):
            if m[l][e] != (g * U + e, i):
                return False
    return True


@pytest.mark.parametrize("U", [2, 4, 8])
def test_butterfly_transposes(U):
    m = butterfly(U)
    assert xpose_ok(U, m)
    # store e: the U lanes of group g write units 0..U-1 of row g*U + e, contiguous
    for e in range(U):
        rows = {}
        for l in range(32):
            g, i = divmod(l, U)
            rows.setdefault(g * U + e, []).append((l, i))
        for row, lanes in rows.items():
            assert sorted(i for _, i in lanes) == list(range(U))
            assert [i for _, i in sorted(lanes)] == list(range(U))  # ascending lanes, ascending units


@pytest.mark.parametrize("U", [2, 4, 8])
def test_butterfly_wrong_partner_caught(U):
    # partner l + s instead of l ^ s (wraps across groups)
    assert not xpose_ok(U, butterfly(U, partner=lambda l, s: (l + s) % 32))


def stage_addr(r, u, xor=True):
    return r * 128 + (((u ^ (r & 7)) if xor else u) << 4)


def conflict_free(addrs):
    """addrs: 32 byte addresses of one 16-byte-per-lane shared access."""
    for phase in range(4):
        groups = {(a // 16) % 8 for a in addrs[8 * phase: 8 * phase + 8]}
        if len(groups) != 8:
            return False
    return True


def test_staging_buffer_conflict_free_and_complete():
    for u in range(8):  # row-wise writes: lane = row, unit u
        assert conflict_free([stage_addr(l, u) for l in range(32)])
    seen = set()
    for k in range(8):  # column-wise reads: lane l reads unit l % 8 of row 4k + l / 8
        addrs = [stage_addr(4 * k + l // 8, l % 8) for l in range(32)]
        assert conflict_free(addrs)
        # 8 lanes of a row read its 8 units: 128 contiguous global bytes
        for l in range(32):
            seen.add((4 * k + l // 8, l % 8))
    assert seen == {(r, u) for r in range(32) for u in range(8)}
    assert len({stage_addr(r, u) for r in range(32) for u in range(8)}) == 256  # a bijection


def test_staging_without_xor_caught():
    assert not conflict_free([stage_addr(l, 0, xor=False) for l in range(32)])
