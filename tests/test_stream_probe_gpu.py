"""The stream probe (dopt_stream_probe), the measurement kernel behind the
read/write-mix ceilings: every write stream receives, at vector i, the XOR
of the read streams' vector i with the seed (i mod 2^32, i >> 32,
0x9e3779b9, 0x7f4a7c15), and a read-only mix writes nothing."""
import pytest
import torch

from zero_distributed_optimizer_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _seed(n):
    i = torch.arange(n, dtype=torch.int64, device=DEV)
    s = torch.empty(n, 4, dtype=torch.int64, device=DEV)
    s[:, 0] = i & 0xFFFFFFFF
    s[:, 1] = i >> 32
    s[:, 2] = 0x9E3779B9
    s[:, 3] = 0x7F4A7C15
    return s


@pytest.mark.parametrize("reads,writes", [(1, 1), (3, 2), (0, 2), (8, 1), (1, 7), (16, 16)])
def test_probe_writes_the_xor_of_its_reads(reads, writes):
    n = 5000 * 16 + 7  # vectors: several blocks and a ragged last one
    g = torch.Generator(device=DEV).manual_seed(reads * 31 + writes)
    rb = [torch.randint(-2 ** 31, 2 ** 31 - 1, (n * 4,), dtype=torch.int32, device=DEV, generator=g)
          for _ in range(reads)]
    wb = [torch.zeros(n * 4, dtype=torch.int32, device=DEV) for _ in range(writes)]
    B.dopt_stream_probe(rb, wb)
    torch.cuda.synchronize()
    want = _seed(n)
    for r in rb:
        want ^= r.view(n, 4).to(torch.int64) & 0xFFFFFFFF
    for w in wb:
        assert torch.equal(w.view(n, 4).to(torch.int64) & 0xFFFFFFFF, want)


def test_probe_read_only_mix_leaves_its_buffers():
    n = 4096
    rb = [torch.full((n * 4,), i + 1, dtype=torch.int32, device=DEV) for i in range(4)]
    before = [r.clone() for r in rb]
    B.dopt_stream_probe(rb, [])
    torch.cuda.synchronize()
    for r, b in zip(rb, before):
        assert torch.equal(r, b)
