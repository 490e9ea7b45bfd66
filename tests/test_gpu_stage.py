"""pks_stage_copy: byte ranges between page-locked host memory and the device
(and device to device) in one launch, 16-byte and byte paths, empty ranges,
eight ranges at once, and replay inside a CUDA graph.  The expected bytes are
the source tensors themselves."""

import numpy as np
import pytest
import torch

from top_sparse_attention_pks_gb300 import build, pks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _host(n, seed):
    g = np.random.default_rng(seed)
    return torch.from_numpy(g.integers(0, 256, size=n, dtype=np.uint8)).pin_memory()


@pytest.mark.parametrize("sizes", [[262144, 8192, 64, 131072], [12, 1, 0, 4096 + 7], [1 << 20]])
def test_host_to_device_and_back(sizes):
    src = [_host(n, i) for i, n in enumerate(sizes)]
    dev = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in sizes]
    back = [torch.zeros(n, dtype=torch.uint8).pin_memory() for n in sizes]
    s = torch.cuda.current_stream()
    pks.pks_stage_copy(list(zip(dev, src)), s)
    pks.pks_stage_copy(list(zip(back, dev)), s)
    torch.cuda.synchronize()
    for a, d, b in zip(src, dev, back):
        assert torch.equal(d.cpu(), a)
        assert torch.equal(b, a)


def test_unaligned_offsets_and_device_to_device():
    a = _host(5000, 7)
    d = torch.zeros(5000, dtype=torch.uint8, device="cuda")
    # a 16-byte aligned size at an odd offset takes the byte path
    pks.pks_stage_copy([(d[3:3 + 4096], a[1:1 + 4096])])
    e = torch.zeros(5000, dtype=torch.uint8, device="cuda")
    pks.pks_stage_copy([(e, d)])
    torch.cuda.synchronize()
    ref = torch.zeros(5000, dtype=torch.uint8)
    ref[3:3 + 4096] = a[1:1 + 4096]
    assert torch.equal(d.cpu(), ref)
    assert torch.equal(e.cpu(), ref)


def test_eight_ranges_of_typed_tensors():
    g = torch.Generator().manual_seed(3)
    srcs = [torch.randn(17 * (i + 1), generator=g).to(torch.bfloat16).pin_memory() for i in range(4)]
    srcs += [torch.randint(-5, 5, (33 * (i + 1),), dtype=torch.int32, generator=g).pin_memory()
             for i in range(4)]
    dsts = [torch.empty_like(x, device="cuda") for x in srcs]
    pks.pks_stage_copy(list(zip(dsts, srcs)))
    torch.cuda.synchronize()
    for x, y in zip(srcs, dsts):
        assert torch.equal(y.cpu(), x)


def test_replay_in_a_cuda_graph_reads_the_host_buffer_each_time():
    h = _host(262144, 11)
    d = torch.empty(262144, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pks.pks_stage_copy([(d, h)], s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pks.pks_stage_copy([(d, h)], s)
    for seed in (12, 13):
        h.copy_(_host(262144, seed))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(d.cpu(), h)


def test_rejects_unpinned_host_tensors_and_size_mismatch():
    d = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        pks.pks_stage_copy([(d, torch.zeros(64, dtype=torch.uint8))])
    with pytest.raises(ValueError):
        pks.pks_stage_copy([(d, _host(32, 1))])
