"""Per-token tensors (qkv, g, beta, gate, slot_idx, out) in pinned host
memory, read and written by the kernel directly over the CPU-GPU link; state,
conv state and weights stay on the GPU.  Same tolerances as the other
parity tests."""
import numpy as np
import pytest
import torch

import kda_testlib as T
from linear_attention_decode_04_gb300 import KdaDecodeCall
from linear_attention_decode_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["n4_h12_pool8", "n32_h24_pool64_pad8", "n128_h48_pool512_normoff"])
@pytest.mark.parametrize("early_prefetch", [False, True])
def test_token_tensors_in_pinned_host_memory(name, early_prefetch, cuda_device):
    x = W.make_inputs(W.SPECS[name])
    d = T.to_device(x, cuda_device)
    h = {k: d[k].cpu().pin_memory() for k in ("qkv", "g", "beta", "gate", "slot_idx")}
    out = torch.full((x.N, x.H * 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    call = KdaDecodeCall(h["qkv"], d["conv_weight"], d["conv_state"], d["state"], h["g"], h["beta"],
                         h["slot_idx"], out, gate=h["gate"], norm_weight=d["norm_weight"], eps=x.spec.eps,
                         out_norm=x.spec.out_norm, err_flag=d["err_flag"], early_prefetch=early_prefetch,
                         host_token_io=True)
    call()
    torch.cuda.synchronize()
    d["out"] = out
    ref = T.run_oracle(x)
    T.compare_all(x, d, ref, init_state=x.state, init_conv=x.conv_state)
    assert int(d["err_flag"].item()) == 0


def test_unpinned_host_tensor_is_refused(cuda_device):
    x = W.make_inputs(W.PR1_REF)
    d = T.to_device(x, cuda_device)
    with pytest.raises(ValueError):
        KdaDecodeCall(d["qkv"].cpu(), d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                      d["slot_idx"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"],
                      host_token_io=True)
