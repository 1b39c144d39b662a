"""The host-buffer backward (binding.HostBackward): copies of one run of GQA
groups overlap the kernels of the previous run, each run being one attn_bwd
call on pointer offsets.  Its gradients must be bitwise those of a single
attn_bwd on device-resident inputs (heads are independent and every kernel
reduces in a fixed order), for several chunk counts and for a block mask
sliced per run, with equal and with uneven runs; with B > 1 the call is not split."""
import pytest
import torch

from masked_attention_backward_gb300 import binding as mab
from masked_attention_backward_gb300.workloads import (MASK_BLOCK, MASK_CAUSAL, MASK_SLIDING,
                                                        Workload, make_inputs)
from parity import forward_stats, gpu_mask

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("pipe_causal_sink_bf16", "bf16", B=1, Hq=8, Hkv=4, Sq=384, Skv=384,
              mask_kind=MASK_CAUSAL, sink=True, seed=81), [1, 2, 4, [1, 2, 1], [3, 1]]),
    (Workload("pipe_blocks_f16", "f16", B=1, Hq=4, Hkv=2, Sq=333, Skv=290, mask_kind=MASK_BLOCK,
              bx=48, by=80, block_pattern="random", density=0.4, sink=True, seed=82), [2]),
    (Workload("pipe_swa_b2_bf16", "bf16", B=2, Hq=4, Hkv=2, Sq=300, Skv=300,
              mask_kind=MASK_SLIDING, window=90, sink=True, seed=83), [2]),
]


@pytest.mark.parametrize("wl,chunk_list", CASES, ids=[c[0].name for c in CASES])
def test_host_pipeline_matches_device_call(cuda_lib, wl, chunk_list):
    inp = make_inputs(wl)
    O, lse = forward_stats(wl, inp)
    dev = torch.device("cuda")
    d = {"q": inp.q.to(dev), "k": inp.k.to(dev), "v": inp.v.to(dev), "o": O.to(dev),
         "dO": inp.dO.to(dev), "lse": lse.to(dev)}
    sink = inp.sink.to(dev) if inp.sink is not None else None
    mask = gpu_mask(wl, inp)
    ref = mab.bwd(d["q"], d["k"], d["v"], d["o"], d["dO"], d["lse"], sink, mask, wl.scale)
    torch.cuda.synchronize()
    host_in = {n: t.cpu().pin_memory() for n, t in d.items()}
    host_in["sink"] = inp.sink.pin_memory() if inp.sink is not None else None
    for chunks in chunk_list:
        host_out = [torch.full_like(t, float("nan")).cpu().pin_memory() if t is not None else None
                    for t in ref]
        hb = mab.HostBackward(wl.B, wl.Hq, wl.Hkv, wl.Sq, wl.Skv, d["q"].dtype, mask, wl.scale,
                              sink is not None, dev, chunks=chunks)
        runs = chunks if isinstance(chunks, list) else [wl.Hkv // chunks] * chunks
        assert hb.sizes == ([wl.Hkv] if wl.B > 1 else runs)
        for _ in range(2):  # twice: nothing may depend on what the previous call left
            hb(host_in, host_out)
            torch.cuda.synchronize()
            for name, a, b in zip(("dq", "dk", "dv", "dsink"), host_out, ref):
                if b is None:
                    continue
                assert torch.equal(a, b.cpu()), f"{wl.name} chunks={chunks}: {name} differs"
