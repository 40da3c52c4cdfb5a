"""The library's bandwidth probes (store, bulk store and copy kernels that
give the codec's store patterns their HBM ceilings) run, write what they
claim to write, and report sensible bandwidths on a buffer beyond L2."""
import pytest
import torch

import agent_shared_compressed_gb300 as kv
from agent_shared_compressed_gb300 import build as kvbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    kvbuild.build()
    kv.load()


def test_probes_write_the_whole_buffer_and_copy_exactly():
    n = (64 << 20) + 4096 * 3                       # ragged against the grid, a multiple of 4 KB
    st = torch.cuda.current_stream()
    guard = 4096
    buf = torch.zeros(n + guard, dtype=torch.uint8, device="cuda")
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_STORE, buf, None, n, st) == kv.KVP_OK
    torch.cuda.synchronize()
    words = buf[:n].view(torch.int32).view(-1, 4)
    assert bool((words[:, 2] == 0x5A5A5A5A).all())  # every 16-byte chunk written
    assert bool((buf[n:] == 0).all())               # nothing past the end
    buf.zero_()
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_BULK_STORE, buf, None, n, st) == kv.KVP_OK
    torch.cuda.synchronize()
    words = buf[:n].view(torch.int32).view(-1, 4)
    assert bool((words[:, 3] == 0x5A5A5A5A).all())
    assert bool((buf[n:] == 0).all())
    src = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")
    dst = torch.zeros(n + guard, dtype=torch.uint8, device="cuda")
    assert kv.kvp_bandwidth_probe(kv.KVP_PROBE_COPY, dst, src, n, st) == kv.KVP_OK
    torch.cuda.synchronize()
    assert torch.equal(dst[:n], src) and bool((dst[n:] == 0).all())


def test_store_ceiling_is_in_a_plausible_range():
    n = 2 << 30
    st = torch.cuda.current_stream()
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    for mode in (kv.KVP_PROBE_STORE, kv.KVP_PROBE_BULK_STORE):
        for _ in range(2):
            assert kv.kvp_bandwidth_probe(mode, buf, None, n, st) == kv.KVP_OK
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        assert kv.kvp_bandwidth_probe(mode, buf, None, n, st) == kv.KVP_OK
        e1.record(st)
        torch.cuda.synchronize()
        gbs = n / (e0.elapsed_time(e1) * 1e-3) / 1e9
        assert 1000 < gbs < 10000, (mode, gbs)
