"""kda_decode_noalloc, the entry point for callers that cannot allocate device
memory (for example code enqueueing inside a CUDA-graph capture, or a plugin
whose enqueue must not allocate): it keeps the dynamic-schedule work queue in
a static device array inside the library instead of a caller buffer.

Called through the C ABI (ctypes) twice in a row on the same pools, and
compared after each call with kda_decode on an identical copy of the inputs,
with the tolerances of the other parity tests.  Collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_testlib as T
from linear_attention_decode_04_gb300 import KdaDecodeCall, binding
from linear_attention_decode_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(call: KdaDecodeCall, stream: torch.cuda.Stream) -> int:
    lib = binding.load_library()
    fn = lib.kda_decode_noalloc
    fn.argtypes = [ctypes.POINTER(binding.KdaDecodeArgs), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn(ctypes.byref(call.args), ctypes.c_void_p(stream.cuda_stream))


def _call(x, d):
    return KdaDecodeCall(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                         d["slot_idx"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"],
                         eps=x.spec.eps, err_flag=d["err_flag"])


def test_noalloc_matches_kda_decode_on_two_calls(cuda_device):
    # 64 x 24 = 1536 units: beyond each CTA's first ring, so the queue is used
    spec = W.Spec("noalloc_n64_h24_pool80", N=64, H=24, num_slots=80, seed=91, pad_tail=3)
    x = W.make_inputs(spec)
    dA, dB = T.to_device(x, cuda_device), T.to_device(x, cuda_device)
    callA, callB = _call(x, dA), _call(x, dB)
    stream = torch.cuda.current_stream(cuda_device)
    second = W.draw_step_inputs(spec, 1)
    for step in range(2):
        if step == 1:  # new token inputs, same pools: the state carries over
            for d in (dA, dB):
                d["qkv"].copy_(T.bf16_tensor(second["qkv"], cuda_device))
                d["g"].copy_(torch.from_numpy(second["g"]))
                d["beta"].copy_(T.bf16_tensor(second["beta"], cuda_device))
                d["gate"].copy_(T.bf16_tensor(second["gate"], cuda_device))
        callA(stream)
        rc = _noalloc(callB, stream)
        assert rc == 0, binding.load_library().kda_last_error().decode()
        torch.cuda.synchronize(cuda_device)
        assert int(dA["err_flag"].item()) == 0 and int(dB["err_flag"].item()) == 0
        a = W.bf16_bits_to_f32(T.bf16_bits(dA["out"])).astype(np.float64)
        b = W.bf16_bits_to_f32(T.bf16_bits(dB["out"])).astype(np.float64)
        assert np.all(np.isfinite(b))
        assert np.abs(a - b).max() <= T.OUT_ATOL, f"call {step + 1}: output differs"
        assert np.array_equal(T.bf16_bits(dA["conv_state"]), T.bf16_bits(dB["conv_state"])), \
            f"call {step + 1}: conv state differs"
        sa, sb = dA["state"].cpu().numpy(), dB["state"].cpu().numpy()
        for s in range(spec.num_slots):
            T.check_state_slot(sb[s], sa[s], f"call {step + 1} slot {s}")
