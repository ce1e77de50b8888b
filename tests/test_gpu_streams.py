"""Independent calls in flight on several streams (GPU).

A server runs independent batches concurrently, and the benchmark's
`two_streams` and end-to-end figures do the same. The library keeps no
per-call state outside the caller's buffers (the workspace included), so
calls with their own output and workspace buffers, launched alternately on
two or three streams and overlapping on the device, must give exactly the
results the same calls give one at a time on one stream: bit for bit, for
each kernel family (16-head bf16 with the cluster merge and with the
workspace merge, the lean E4M3 kernel, the 128-head kernel with its q
pre-pass)."""
import pytest
import torch

from parity import DEV, gpu_cache
from sparse_mla_attention_04_gb300 import binding

pytestmark = pytest.mark.gpu


def _inputs(T, H, D_qk, topk, slots, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    q = torch.randn(T, H, D_qk, generator=g, device=DEV).to(torch.bfloat16)
    idx = torch.randint(0, slots, (T, topk), generator=g, device=DEV, dtype=torch.int32)
    idx[:, ::5] = -1
    return q, idx


@pytest.mark.parametrize("H,D_qk,fp8,num_splits,lanes", [
    (16, 512, False, 0, 2),     # cluster merge of the automatic plan
    (16, 512, False, 12, 3),    # workspace merge (tickets in the workspace)
    (16, 512, True, 0, 2),      # lean E4M3 kernel, fp8 dots
    (16, 512, False, 1, 3),     # one split per row (the plan for a shared GPU), no merge
    (16, 512, True, 2, 3),      # lean E4M3 kernel, two splits (the plan for a shared GPU)
    (128, 576, True, 0, 2),     # q pre-pass + 128-head kernel
])
def test_concurrent_calls_match_serial(H, D_qk, fp8, num_splits, lanes):
    T, topk, slots, n = 24, 1024, 20000, 6
    g = torch.Generator(device=DEV)
    g.manual_seed(H + D_qk + num_splits)
    kv_src = torch.randn(slots, D_qk, generator=g, device=DEV).to(torch.bfloat16)
    cache, kvs = gpu_cache(kv_src, fp8)
    dot = "fp8" if fp8 else "auto"
    sets = [_inputs(T, H, D_qk, topk, slots, 100 + i) for i in range(n)]
    need = binding.sparse_mla_fwd_ex_workspace_size(T, H, D_qk, 512, topk, 1 if fp8 else 0,
                                                    dot_precision=dot, num_splits=num_splits)

    def run(streams):
        outs = []
        for i, (q, idx) in enumerate(sets):
            st = streams[i % len(streams)]
            out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=DEV)
            lse = torch.empty((T, H), dtype=torch.float32, device=DEV)
            ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=DEV)
            with torch.cuda.stream(st):
                binding.sparse_mla_fwd(q, cache, idx, 0.0625, kv_scale=kvs, dot_precision=dot, out=out, lse=lse,
                                       workspace=ws, num_splits=num_splits, stream=st)
            outs.append((out, lse, ws))
        torch.cuda.synchronize()
        return [(o.cpu(), l.cpu()) for o, l, _ in outs]

    serial = run([torch.cuda.Stream(device=DEV)])
    concurrent = run([torch.cuda.Stream(device=DEV) for _ in range(lanes)])
    for (so, sl), (co, cl) in zip(serial, concurrent):
        assert torch.equal(so, co) and torch.equal(sl, cl)
    assert binding.smla_device_error() == 0
