"""The interference probes (resident-CTA / SM-id probe, bulk-copy read probe) on the GPU."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tide():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import all_gather_tide_gb300 as t

    t.lib()
    return t


def test_hold_probe_records_sm_ids_and_times(tide):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 8
    rec = torch.zeros(3 * n, dtype=torch.int64, device="cuda")
    tide.tide_probe_hold(n, 1024, 213 * 1024, 4, 200_000, rec)
    torch.cuda.synchronize()
    r = rec.view(n, 3).cpu().numpy()
    assert np.all((r[:, 0] >= 0) & (r[:, 0] < sms))
    assert np.all(r[:, 2] - r[:, 1] >= 200_000)
    # each CTA fills an SM, and 8 fit at once: 8 different SMs, all started together
    assert len(set(r[:, 0].tolist())) == n
    assert r[:, 1].max() - r[:, 1].min() < 150_000


def test_bulk_read_probe_checksum(tide):
    nbytes = 256 << 20
    copy = 49152
    buf = torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), dtype=torch.int32, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    tide.tide_probe_bulk_read(buf, nbytes, 16, copy, 4, out)
    torch.cuda.synchronize()
    nchunk = nbytes // copy
    firsts = buf.view(-1)[: nchunk * copy // 4].view(nchunk, copy // 4)[:, 0].cpu().numpy().view(np.uint32)
    want = np.bitwise_xor.reduce(firsts)
    got = out.cpu().numpy().view(np.uint32)
    assert got[1] == 0
    assert got[0] == want


@pytest.mark.parametrize("consumers,ldg_warps", [(15, 0), (0, 0), (8, 7), (1, 14)])
def test_ingest_probe_reads_every_byte(tide, consumers, ldg_warps):
    """The per-SM ingest probe reads all of both parts: its checksum equals the XOR of every 32-bit
    word of the bulk part (or of each copy's first word when the slots are not read out) and of
    every word of the register-load part."""
    copy, stages = 46080, 4
    bulk = (96 << 20) // copy * copy if ldg_warps < 14 else 0
    ldg = (32 << 20) if ldg_warps else 0
    ldg_off = (bulk + 255) // 256 * 256
    words = (ldg_off + ldg) // 4 + 64
    buf = torch.randint(-2**31, 2**31 - 1, (words,), dtype=torch.int32, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    tide.tide_probe_ingest(buf, bulk, ldg, 16, copy, stages, consumers, ldg_warps, out)
    torch.cuda.synchronize()
    h = buf.cpu().numpy().view(np.uint32)
    want = np.uint32(0)
    if bulk:
        part = h[: bulk // 4]
        want ^= np.bitwise_xor.reduce(part if consumers else part.reshape(-1, copy // 4)[:, 0])
    if ldg:
        want ^= np.bitwise_xor.reduce(h[ldg_off // 4: (ldg_off + ldg) // 4])
    got = out.cpu().numpy().view(np.uint32)
    assert got[1] == 0
    assert got[0] == want


def test_mixed_probe_writes_its_pattern_once(tide):
    """Writers alone (no reads): every 32-byte vector of each CTA's share holds the pattern of the
    thread that wrote it, the bytes beyond the shares are untouched, and the count is exact."""
    ctas, st_warps = 16, 4
    nt = st_warps * 32
    st_bytes = (64 << 20) + 96  # shares of whole vectors; 96 bytes left over
    per = st_bytes // 32 // ctas
    st = torch.full((st_bytes // 4 + 64,), -1, dtype=torch.int32, device="cuda")
    src = torch.zeros(1024, dtype=torch.int32, device="cuda")
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    tide.tide_probe_mixed(src, 0, st, st_bytes, ctas, 73728, 3, 1, st_warps, out)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert o[1] == 0 and o[2] == per * 32 * ctas
    w = st.cpu().numpy().view(np.uint32)
    vec = w[: ctas * per * 8].reshape(ctas, per, 8)
    b = np.arange(ctas, dtype=np.uint64)[:, None]
    v = np.arange(per, dtype=np.uint64)[None, :]
    want = ((np.uint64(0x9E3779B9) * (b * np.uint64(1024) + v % np.uint64(nt))) % np.uint64(1 << 32)).astype(np.uint32)
    want ^= v.astype(np.uint32)
    assert np.array_equal(vec, np.repeat(want[:, :, None], 8, axis=2))
    assert np.all(w[ctas * per * 8:] == 0xFFFFFFFF)


@pytest.mark.parametrize("consumers,st_warps", [(15, 0), (11, 4), (14, 1)])
def test_mixed_probe_reads_every_byte_while_writing(tide, consumers, st_warps):
    copy, stages = 73728, 3
    bulk = (96 << 20) // copy * copy
    buf = torch.randint(-2**31, 2**31 - 1, (bulk // 4 + 64,), dtype=torch.int32, device="cuda")
    st = torch.empty(32 << 20, dtype=torch.uint8, device="cuda")
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    tide.tide_probe_mixed(buf, bulk, st, st.numel(), 16, copy, stages, consumers, st_warps, out)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    want = np.bitwise_xor.reduce(buf.cpu().numpy().view(np.uint32)[: bulk // 4])
    assert o[1] == 0
    assert np.uint32(o[0] & 0xFFFFFFFF) == want
    assert (o[2] > 0) == (st_warps > 0)


def test_mixed_probe_burst_writes_count(tide):
    """Reading threads that also write in bursts (the reduce-scatter's store pattern): every byte is
    still read, and the bytes written are exactly the bursts the CTAs' copies call for."""
    copy, stages, cons, ctas, rows, vecs = 46080, 5, 15, 16, 8, 6
    nchunk = (64 << 20) // copy
    bulk = nchunk * copy
    buf = torch.randint(-2**31, 2**31 - 1, (bulk // 4 + 64,), dtype=torch.int32, device="cuda")
    st = torch.empty(16 << 20, dtype=torch.uint8, device="cuda")
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    tide.tide_probe_mixed(buf, bulk, st, st.numel(), ctas, copy, stages, cons, 0, out, burst_rows=rows, burst_vecs=vecs)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    per_cta = [len(range(b, nchunk, ctas)) for b in range(ctas)]
    want_written = sum(k // rows for k in per_cta) * cons * 32 * vecs * 32
    assert o[1] == 0 and o[2] == want_written
    assert np.uint32(o[0] & 0xFFFFFFFF) == np.bitwise_xor.reduce(buf.cpu().numpy().view(np.uint32)[: bulk // 4])
