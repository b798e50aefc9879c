"""A decode step through the C ABI can be captured in a CUDA graph and replayed: the calls do no
host synchronisation and allocate nothing, so a serving loop can replay one captured step per
token. Replays with new inputs written in place must equal eager calls bit for bit."""
import numpy as np
import pytest
import torch

import indexer_top_sparse_paged_gb300 as dsa
import workloads as W
from cases import small_spec
from gpu_helpers import Dev

pytestmark = pytest.mark.gpu


def test_decode_step_replays_from_a_cuda_graph():
    spec = small_spec("bf16", [700, 3000, 5000, 2049], 512)
    case = W.generate(spec, seed=301)
    d = Dev(case)
    idx = torch.empty((spec.T, spec.K), dtype=torch.int32, device="cuda")
    out = torch.empty((spec.T, spec.H, spec.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((spec.T, spec.H), dtype=torch.float32, device="cuda")

    def step():
        dsa.decode(d.dims, d.q_I, d.w, d.k_I, d.k_I_scale, d.block_table, d.seq_lens, d.q, d.kv, spec.sm_scale,
                   ws=d.ws, idx=idx, out=out, lse=lse)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture (first-call set-up of the kernels)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    rng = np.random.default_rng(302)
    for _ in range(2):
        # new queries and head weights, written in place into the captured buffers
        d.q_I.copy_(torch.from_numpy(W.to_bf16_bits(rng.standard_normal(case.q_I.shape, dtype=np.float32)).view(np.int16))
                    .view(torch.bfloat16))
        d.q.copy_(torch.from_numpy(W.to_bf16_bits(rng.standard_normal(case.q.shape, dtype=np.float32)).view(np.int16))
                  .view(torch.bfloat16))
        d.w.copy_(torch.from_numpy(rng.uniform(0, 1, case.w.shape).astype(np.float32)))
        g.replay()
        torch.cuda.synchronize()
        g_idx, g_out, g_lse = idx.clone(), out.clone(), lse.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(g_idx, idx) and torch.equal(g_out, out) and torch.equal(g_lse, lse)
        assert dsa.read_error(d.ws) == 0
