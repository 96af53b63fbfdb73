"""Index arithmetic of the fused compression kernel, checked on the CPU for
every launch shape its dispatch table uses (parsed from the kernel header, so
a new shape is checked as soon as it is added).  Each check restates one
bound the kernel relies on: shared-memory ring and partial-sum buffers, the
lanes that hold chunk totals, the sign-word and error stores of a tile, and
the 16-byte sizes of the bulk copies."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "communication_compressed_optimizer_gb300", "csrc", "k_compress.cuh")
SMEM_PER_BLOCK = 227 * 1024          # opt-in shared memory per CTA on sm_103a
SMEM_PER_SM = 228 * 1024


def dispatched_shapes():
    text = open(HDR).read()
    body = text[text.index("cudaError_t launch_fused_all_chunks"):]
    shapes = set()
    for m in re.finditer(r"launch_grad<(\d+), (\d+), (\d+), (\d+), ADAM, EB>", body):
        nt, slots, nslot, c = map(int, m.groups())
        for gk in (0, 1, 2):
            shapes.add((nt, slots, nslot, c, gk, 0))
    for m in re.finditer(r"launch_one<(\d+), (\d+), kGrad(F32|BF16|Philox), (\d+), (\d+), ADAM, EB(?:, (\d+))?>",
                         body):
        nt, slots, kind, nslot, c, ndraw = m.groups()
        shapes.add((int(nt), int(slots), int(nslot), int(c), {"F32": 0, "BF16": 1, "Philox": 2}[kind],
                    int(ndraw or 0)))
    return sorted(shapes)


SHAPES = dispatched_shapes()


def test_dispatch_table_was_parsed():
    cs = {s[3] for s in SHAPES}
    assert cs == {256, 512, 1024, 2048, 4096, 8192}
    assert (512, 2, 7, 4096, 0, 0) in SHAPES
    assert (512, 2, 7, 4096, 2, 512) in SHAPES        # in-kernel gradients with draw warps


@pytest.mark.parametrize("nt,slots,nslot,c,gk,ndraw", SHAPES)
def test_shape_bounds(nt, slots, nslot, c, gk, ndraw):
    tile = nt * 4 * slots
    nwarp = nt // 32
    npart = tile // 128
    ppc = c // 128
    cpt = tile // c
    assert nt % 32 == 0 and nt <= 1024
    assert tile % c == 0 and cpt >= 1, "a tile holds whole chunks"
    assert slots & (slots - 1) == 0 and slots <= 8, "pack_words handles up to 8 slots"
    # ring: NSLOT slots of TILE floats; two CTAs per SM when two rings fit; a
    # CTA with draw warps adds kDrawSlots gradient tiles and runs alone
    slot_bytes = tile * 4
    draw_slots = 3 if ndraw else 0
    ring = nslot * slot_bytes
    min_blocks = 1 if ndraw else (3 if ring <= 72 * 1024 else (2 if ring <= 112 * 1024 else 1))
    static = 2 * npart * 4 + 64 * 4 + nslot * 8 + 2 * max(draw_slots, 1) * 8 + 4   # red, lmax, mbarriers
    dyn = (nslot + draw_slots) * slot_bytes
    assert dyn + static <= SMEM_PER_BLOCK
    assert min_blocks * (dyn + static + 1024) <= SMEM_PER_SM
    threads = nt + ndraw
    assert threads <= 1024
    assert 65536 // (threads * min_blocks) >= 64 or (min_blocks == 3 and 65536 // (threads * 3) >= 80), \
        "the launch bound leaves at least 64 registers (80 at three CTAs of 256)"
    if ndraw:
        assert gk == 2, "draw warps only for in-kernel gradients"
        assert ndraw % 32 == 0 and nt % 32 == 0      # whole warps: per-warp arrivals, named barrier 1
        pg = tile // (4 * ndraw)
        assert pg >= 1 and pg * 4 * ndraw == tile
        groups = set()
        for d in range(ndraw):
            for g in range(pg):
                e = g * ndraw * 4 + d * 4
                assert 0 <= e and e + 4 <= tile
                groups.add(e)
        assert len(groups) == tile // 4, "every group of four of the tile is drawn exactly once"
    # the 128-leaf partial of slot s, warp w is red[s * NWARP + w], in element order
    for s in range(slots):
        for w in range(nwarp):
            idx = s * nwarp + w
            assert idx < npart and idx * 128 == s * nt * 4 + w * 128
    # chunk totals: G partials per lane (one vector load), LPC lanes per chunk
    g = 4 if ppc >= 4 else ppc
    lpc = ppc // g
    lused = npart // g
    assert ppc % g == 0 and lused * g == npart and 1 <= lused <= 32
    assert (npart * 4) % 16 == 0, "red[1] stays 16-byte aligned for the vector loads"
    for lane in range(32):
        lq = lane % lused
        assert lq * g + g <= npart
        assert lq // lpc < cpt                                   # a chunk of this tile
    # the lane holding a slot's chunk scale (qsrc) is one with that chunk's total
    for s in range(slots):
        for w in range(nwarp):
            chunk = (s * nt * 4 + w * 128) // c
            src = chunk * lpc
            assert src < lused and (src % lused) // lpc == chunk
    # sign words: lanes with (lane & 7) < SLOTS store word (lane >> 3) of slot
    # tree_block(lane), all inside the tile's TILE/32 words
    def tree_block(lane):
        b, o, n = 0, 1, slots
        while n > 1:
            if lane & o:
                b += n // 2
            n //= 2
            o <<= 1
        return b
    words = set()
    for w in range(nwarp):
        for lane in range(32):
            if (lane & 7) < slots:
                wd = (w * 128) // 32 + (lane >> 3) + tree_block(lane) * (nt * 4 // 32)
                assert 0 <= wd < tile // 32
                words.add(wd)
    assert len(words) == tile // 32, "every word of the tile is stored exactly once per warp set"
    # error stores: thread tid writes 4 elements at s*NT*4 + tid*4 inside the tile
    assert (slots - 1) * nt * 4 + (nt - 1) * 4 + 4 <= tile
    # bulk copies: slot-sized copies and the packed-momentum words are 16-byte multiples
    assert slot_bytes % 16 == 0 and (tile // 8) % 16 == 0
    grad_bytes = {0: 4, 1: 2, 2: 0}[gk]
    if grad_bytes:
        assert (tile * grad_bytes) % 16 == 0
        # a partial last tile copies (N - base) gradients rounded up to 16 bytes: inside a row of
        # the smallest leading dimension the API accepts (ld >= N, ld * bytes a multiple of 16)
        per16 = 16 // grad_bytes
        for n in range(1, 2 * tile + 40):
            ld = -(-n // per16) * per16
            base = (n - 1) // tile * tile
            copied = -(-(n - base) * grad_bytes // 16) * 16
            assert base * grad_bytes + copied <= ld * grad_bytes, n
    # scale span of the packed momentum: from k0 & ~3, (k0 & 3) + CPT floats rounded up to 16
    # bytes, for every tile of the padded length, never past scale_s[K + 16) (the region has 16
    # floats of padding), and it fits in the momentum slot after the tile's sign words
    step = max(c, 4096)
    for n in list(range(1, 3 * step + 2, 97)) + [step * k + d for k in (1, 2, 5) for d in (-1, 0, 1)]:
        k = -(-n // c)
        npad = -(-n // step) * step
        for t in range(npad // tile):
            k0 = t * tile // c
            ka = k0 & ~3
            sbytes = ((k0 - ka + cpt) * 4 + 15) // 16 * 16
            assert ka + sbytes // 4 <= k + 16, (n, t)
            assert tile // 8 + sbytes <= slot_bytes


def _ring_schedule(W, nslot, adam, late, ntiles, per_worker=2):
    """The fused kernel's copy-ring schedule, restated: thread 0 issues items
    in order while their slots fit ahead of the released positions; the
    compressing threads wait for an item's slots, and release them after the
    barrier that follows their last read.  Items per tile: M (1 slot), W
    workers (gradients + errors, 2 slots each; errors only, 1 slot, when the
    gradients are drawn in the kernel), the server's S (errors, and
    for 1-bit LAMB the frozen preconditioner: 1 or 2 slots) and, for 1-bit
    LAMB, F (old fresh variance, 1 slot).  With late server reads the
    preconditioner and F slots are released only at the end of the tile.
    Returns the number of waits; fails if a wait is for slots not yet issued
    (the kernel would wait for a copy that no thread will issue) or a slot is
    released before it was read."""
    kserver = 1 if adam else 2
    n_items = W + (2 if adam else 3)

    def slots(r):
        return 1 if r == 0 else (per_worker if r <= W else (kserver if r == W + 1 else 1))

    st = dict(issue_pos=0, released=0, tile=0, r=0, cp=0, waits=0)

    def issue_ready():
        while st["tile"] < ntiles:
            n = slots(st["r"])
            if st["issue_pos"] + n > st["released"] + nslot:
                break
            st["issue_pos"] += n
            st["r"] += 1
            if st["r"] == n_items:
                st["r"], st["tile"] = 0, st["tile"] + 1

    def wait(n):
        assert st["cp"] + n <= st["issue_pos"], "waits for slots no thread will issue"
        st["cp"] += n
        st["waits"] += 1

    def release(n):
        st["released"] += n
        assert st["released"] <= st["cp"], "released before it was read"
        issue_ready()

    issue_ready()
    for _ in range(ntiles):
        wait(1)                                         # M
        for w in range(W):
            wait(per_worker)
            release(1 + per_worker if w == 0 else per_worker)   # after the worker's barrier
        nsrv = kserver + (0 if adam else 1)
        wait(nsrv)
        release(1 if late else nsrv)                    # after the server's barrier
        if late:
            release(2)                                  # end of the tile
    assert st["released"] == st["cp"] == st["issue_pos"]
    return st["waits"]


@pytest.mark.parametrize("W", [1, 2, 3, 16, 32])
@pytest.mark.parametrize("nslot,adam,late,per_worker", [
    (7, False, False, 2), (7, True, False, 2), (4, True, False, 2), (4, False, True, 2),
    (4, False, False, 2), (7, False, True, 1), (7, True, False, 1)])
def test_ring_schedule_never_waits_for_an_unissued_copy(W, nslot, adam, late, per_worker):
    assert _ring_schedule(W, nslot, adam, late, ntiles=5, per_worker=per_worker) == 5 * (W + 2)


def test_ring_schedule_check_has_teeth():
    # a ring too small for the server's three slots cannot be scheduled
    with pytest.raises(AssertionError):
        _ring_schedule(4, 2, False, False, ntiles=2)
    # holding all three server slots to the end of the tile needs them free
    # ahead of the next tile's first worker: fine with 4 slots, and the late
    # release of two slots is what the LAMB three-CTA shape uses
    assert _ring_schedule(4, 3, False, True, ntiles=3) == 3 * 6


def test_late_server_reads_fit_the_ring():
    text = open(HDR).read()
    assert "constexpr bool LATE = !ADAM && !WIDE4096;" in text
    for nt, slots, nslot, c, gk, ndraw in SHAPES:
        # the server holds S, D and F (three slots) until the end of the tile,
        # and the next tile's momentum slot must fit beside them
        assert nslot >= 4
        per_worker = 1 if gk == 2 else 2
        for W in (1, 2, 16, 33):
            _ring_schedule(W, nslot, False, True, ntiles=3, per_worker=per_worker)
