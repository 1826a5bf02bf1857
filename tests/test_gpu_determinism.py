"""The results of a call depend on its inputs only: every output, workspace and
saved-context buffer the API allocates is written before it is read.  The
bench's exact calls (forward keeping its context, backward reading it; the
forward alone) run twice, once with every buffer the library's Python layer
allocates filled with zero bytes and once with 0xFF bytes (NaN in every float
format), and must agree bit for bit."""
import contextlib

import pytest
import torch

import bench
import gdn_synth
from gpu_helpers import lib

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def filled_allocations(byte):
    """torch.empty returns CUDA buffers whose bytes are all `byte` (only the
    library's calls run inside)."""
    real = torch.empty

    def empty(*shape, **kw):
        t = real(*shape, **kw)
        if t.is_cuda and t.numel() > 0:
            t.view(torch.uint8).fill_(byte)
        return t

    torch.empty = empty
    try:
        yield
    finally:
        torch.empty = real


def _run(step, p, l2, byte):
    gdn = lib()
    d = p.to("cuda")
    torch.cuda.synchronize()
    with filled_allocations(byte):
        res = step(gdn, d, p.meta["cp"], l2)
        torch.cuda.synchronize()
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    return [t.cpu() for t in res if t is not None]


@pytest.mark.parametrize("name,kw", [
    ("edge", dict(T=4096)),                                  # sequence parallelism forced
    ("training", dict(B=1, T=1024, H=128)),                  # fused walks
    ("varlen", dict(lengths=[700, 0, 64, 1333, 1], H=32)),   # varlen, fused walks
])
@pytest.mark.parametrize("l2", [False, True])
def test_step_does_not_depend_on_buffer_contents(name, kw, l2):
    p = gdn_synth.make(name, **kw)
    for step in (bench.training_step, bench.forward_step):
        a = _run(step, p, l2, 0x00)
        b = _run(step, p, l2, 0xFF)
        assert len(a) == len(b)
        for i, (x, y) in enumerate(zip(a, b)):
            assert torch.isfinite(x.float()).all(), (step.__name__, i)
            assert torch.equal(x, y), (step.__name__, i, (x.float() - y.float()).abs().max())


@pytest.mark.parametrize("l2", [False, True])
def test_repeated_steps_are_bit_identical(l2):
    """The same step, twenty times: any ordering race between the kernels' warps
    shows as a difference (128 walks and 152 persistent local-gradient CTAs,
    each ending on its own last item)."""
    gdn = lib()
    p = gdn_synth.make("training", B=1, T=1024, H=128)
    d = p.to("cuda")
    ref = [t.clone() for t in bench.training_step(gdn, d, p.meta["cp"], l2) if t is not None]
    for rep in range(20):
        if rep % 2:
            bench.forward_step(gdn, d, p.meta["cp"], not l2)      # other kernels in between
        out = [t for t in bench.training_step(gdn, d, p.meta["cp"], l2) if t is not None]
        torch.cuda.synchronize()
        for i, (x, y) in enumerate(zip(ref, out)):
            assert torch.equal(x, y), (rep, i, (x.float() - y.float()).abs().max())
