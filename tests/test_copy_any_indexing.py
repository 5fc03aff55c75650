"""Index arithmetic of the placement kernels' any-alignment run copy, on the CPU.

`copy_bf16_any_alignment` (all_gather_tide_gb300/csrc/copy_any.cuh) copies a run of bf16 elements
between addresses of any alignment: a head of elements aligns the destination to 16 bytes, then
either plain 16-byte vectors (source aligned too) or 16-byte stores assembled from the two aligned
16-byte source words each one straddles, reading only words that lie wholly inside the run; the
rest goes element by element.  This test restates that arithmetic and checks, for every pair of
address alignments and many run lengths, that every element is written exactly once, that every
16-byte word read lies inside the run, and that the assembled bytes are the right ones.  The GPU
parity tests check the kernels' output itself.
"""
import itertools


def plan_copy(da: int, sa: int, n: int):
    """(elements written per index, aligned source words read, byte offset of the shifted path)."""
    head = min(((16 - (da & 15)) & 15) // 2, n)
    s = sa + 2 * head
    s_off = s & 15
    written = [0] * n
    reads = []
    lo = hi = head
    if s_off == 0:
        nv = (n - head) // 8
        for i in range(nv):
            for e in range(8):
                written[head + 8 * i + e] += 1
        hi = head + 8 * nv
    else:
        base = s - s_off
        iend = (s_off + 2 * (n - head)) // 16 - 1
        if iend >= 2:
            lo, hi = head + 8, head + 8 * iend
            for i in range(1, iend):
                reads.append((base + 16 * i, base + 16 * (i + 1)))
                for e in range(8):
                    written[head + 8 * i + e] += 1
    for k in itertools.chain(range(0, lo), range(hi, n)):
        written[k] += 1
    return written, reads, s_off, head


def bytes_at(a: bytes, b: bytes, off: int) -> bytes:
    """The device helper's selection: whole 32-bit words skipped, then a 16-bit funnel shift."""
    c = [int.from_bytes((a + b)[4 * j:4 * j + 4], "little") for j in range(8)]
    q = off >> 2
    o = [c[j + q] for j in range(5)]
    if off & 2:
        o = [((o[j] >> 16) | (o[j + 1] << 16)) & 0xFFFFFFFF for j in range(4)] + [o[4]]
    return b"".join(x.to_bytes(4, "little") for x in o[:4])


def test_every_element_once_and_reads_inside_the_run():
    for da, sa in itertools.product(range(0, 32, 2), repeat=2):
        for n in list(range(0, 70)) + [255, 256, 1000, 8192]:
            dst, src = 4096 + da, 65536 + sa
            written, reads, _, head = plan_copy(dst, src, n)
            assert all(w == 1 for w in written), (da, sa, n)
            for lo, hi in reads:
                assert lo % 16 == 0 and src + 2 * head <= lo and hi <= src + 2 * n, (da, sa, n, lo)


def test_shifted_stores_carry_the_right_bytes():
    memory = bytes((i * 37 + 11) & 0xFF for i in range(4096))
    for off in range(2, 16, 2):
        for i in range(0, 4000 - 32, 16):
            a, b = memory[i:i + 16], memory[i + 16:i + 32]
            assert bytes_at(a, b, off) == memory[i + off:i + off + 16], (off, i)
