"""The C-ABI calls inside a CUDA graph, as a serving loop captures a decode
step: the context-KV write (weight-streaming kernel and CTA pairs with the
split-first schedule, whose arrival counters reset themselves) and the draft
attention (split kernel, then the merge as a programmatic dependent launch).

Each call is captured once with torch.cuda.graph after an eager warm-up on
the same buffers; replaying the graph must give the eager call's bits, also
after the inputs were rewritten in place (the graph reads the buffers, not
values frozen at capture).  The eager results themselves are checked against
the oracle by the parity tests.
"""
import numpy as np
import pytest

import synthetic
from synthetic.device import bits_to_tensor, make_pools, stage

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from draft_model_kv_gb300 import build
    build.build()


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("tokens", [64, 512], ids=["stream-64", "pairs-512"])
def test_write_replays_in_a_cuda_graph(tokens):
    import draft_model_kv_gb300 as dk
    w = synthetic.make_workload("decode512", tokens=tokens)
    st = stage(w)
    bundle = dk.dspark_pack_ctx_kv(st["layers"], w.H)
    eager_pools = dk.dspark_bind_pools(bundle, st["k_pools"], st["v_pools"])
    graph_pools_list = make_pools(w, "cuda")
    graph_pools = dk.dspark_bind_pools(bundle, graph_pools_list[0::2], graph_pools_list[1::2])
    x = st["ctx_hidden"].clone()

    def write(pools):
        dk.dspark_write_ctx_kv(bundle, x, st["positions"], st["cos_sin"], st["cache_loc"], pools,
                               commit_lens=st["commit_lens"], loc_row_width=st["loc_row_width"])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        write(graph_pools)                      # warm-up on the capture buffers
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        write(graph_pools)
    for round_ in range(2):
        if round_ == 1:
            # new hidden states in place: the replay must read them
            x.copy_(torch.flip(st["ctx_hidden"], dims=[0]))
        write(eager_pools)
        g.replay()
        torch.cuda.synchronize()
        assert dk.dspark_get_device_status(bundle) == 0
        for a, b in zip(list(st["k_pools"]) + list(st["v_pools"]),
                        graph_pools_list[0::2] + graph_pools_list[1::2]):
            assert _same_bits(a, b), f"round {round_}"
    bundle.free()


def test_attention_replays_in_a_cuda_graph():
    import draft_model_kv_gb300 as dk
    # several context splits per request, so the merge kernel has work
    a = synthetic.make_attention_workload(3, 8, 32, 8, 128, 2500, 5000)
    dt = torch.bfloat16
    t = lambda v: bits_to_tensor(v, dt, "cuda")
    q, ke, ve, kp, vp = t(a.q), t(a.k_ext), t(a.v_ext), t(a.k_pool), t(a.v_pool)
    idx = torch.from_numpy(a.kv_indices).cuda()
    start = torch.from_numpy(a.kv_start).cuda()
    nbytes = dk.dspark_draft_attention_workspace_bytes(a.batch, a.block, a.num_q_heads, a.num_kv_heads, a.D,
                                                       a.max_context)
    work = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_g = torch.empty_like(q)

    def attend(out, workspace):
        return dk.dspark_draft_attention(q, ke, ve, kp, vp, idx, start, a.sm_scale, a.max_context, out=out,
                                         workspace=workspace, status_flags=status)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        attend(out_g, work)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attend(out_g, work)
    rng = np.random.default_rng(5)
    for round_ in range(2):
        if round_ == 1:
            q.copy_(torch.from_numpy(rng.standard_normal(tuple(q.shape)).astype(np.float32)).to(dt).cuda())
        out_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        eager = attend(None, None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert _same_bits(out_g, eager), f"round {round_}"
