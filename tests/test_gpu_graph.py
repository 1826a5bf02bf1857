"""CUDA-graph capture of the public API: every call launches only on the
current stream and neither allocates nor synchronises inside the library, so
a forward + backward step captured once replays to the same results as the
eager calls (bit for bit: the kernels use no atomics and a fixed reduction
order), with intra-card sequence parallelism on and off."""
import numpy as np
import pytest
import torch

import gdn_synth
from gpu_helpers import lib, to_np

pytestmark = pytest.mark.gpu


def _step(gdn, x, cp):
    o, fs, saved = gdn.chunk_gated_delta_rule_fwd(x.q, x.k, x.v, x.g, x.beta, initial_state=x.h0,
                                                  output_final_state=True, cu_seqlens=x.cu_seqlens,
                                                  cp=cp, save_ctx=True)
    grads = gdn.chunk_gated_delta_rule_bwd(x.q, x.k, x.v, x.g, x.beta, x.do, dht=x.dht,
                                           initial_state=x.h0, cu_seqlens=x.cu_seqlens, cp=cp,
                                           ctx=saved)
    return (o, fs) + tuple(grads)


@pytest.mark.parametrize("cp", ["off", "force"])
def test_graph_replay_matches_eager(cp):
    gdn = lib()
    p = gdn_synth.make("training", B=1, T=1000, H=2, h0_std=0.1, dht_std=0.01)
    d = p.to("cuda")
    eager = [to_np(t) for t in _step(gdn, d, cp) if t is not None]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(gdn, d, cp)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = _step(gdn, d, cp)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert gdn.gdn_sync_status(torch.cuda.current_stream().cuda_stream) == 0
    replayed = [to_np(t) for t in outs if t is not None]
    assert len(replayed) == len(eager)
    for a, b in zip(eager, replayed):
        np.testing.assert_array_equal(a, b)
