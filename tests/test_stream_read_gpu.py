"""rf_stream_read, the read-bandwidth probe: its XOR checksum must equal the
XOR of every 32-bit word of the buffer, computed on the host, for sizes
around its block and unroll boundaries and for a buffer large enough to
take the grid-stride loop several times."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def host_xor(t):
    w = t.cpu().contiguous().view(torch.int32).reshape(-1).numpy().view(np.uint32)
    return int(np.bitwise_xor.reduce(w, dtype=np.uint32)) if w.size else 0


@pytest.mark.parametrize("n16", [1, 3, 255, 1024, 1025, 4096 * 37 + 5, (1 << 22) + 17])
def test_checksum_matches_host(rf, n16):
    g = torch.Generator().manual_seed(n16)
    x = torch.randint(-2**31, 2**31 - 1, (n16 * 4,), generator=g, dtype=torch.int32).cuda()
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    rf.rf_stream_read(x, out)
    torch.cuda.synchronize()
    assert (int(out.item()) & 0xffffffff) == host_xor(x)
    # a second call XORs the same value in again: back to zero
    rf.rf_stream_read(x, out)
    torch.cuda.synchronize()
    assert int(out.item()) == 0


def test_routing_logits_floor_input(rf):
    import synthetic_inputs as si
    x = si.routing_logits(16384, 256, seed=3).cuda()
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    rf.rf_stream_read(x, out)
    torch.cuda.synchronize()
    assert (int(out.item()) & 0xffffffff) == host_xor(x)
