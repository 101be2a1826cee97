"""kda_decode_noalloc, the entry point for callers that cannot allocate device
memory (a plugin whose enqueue step must not allocate, a serving loop with a
memory budget fixed at start-up, a caller that holds no device allocator of
its own): it keeps the dynamic-schedule work queue in a static device array
inside the library instead of a caller buffer.

Called through the C ABI (ctypes) twice in a row on the same pools.  After
each call its output, state and conv state are compared with the fp64 oracle
(chained over the two calls, at the decode tolerances) and with kda_decode
run on an identical copy of the inputs.

The file is named so that pytest collects it after every other test file:
a run that stops at the first failure (-x) has then run all the other tests
before this one.  Nothing else depends on the order; the test also passes
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import kda_testlib as T
import oracle
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


def test_noalloc_matches_oracle_and_kda_decode_on_two_calls(cuda_device):
    # 64 x 24 = 1536 units: beyond each CTA's first ring, so the queue is used
    spec = W.Spec("noalloc_n64_h24_pool80", N=64, H=24, num_slots=80, seed=91, pad_tail=3)
    x = W.make_inputs(spec)
    dA, dB = T.to_device(x, cuda_device), T.to_device(x, cuda_device)
    callA, callB = _call(x, dA), _call(x, dB)
    stream = torch.cuda.current_stream(cuda_device)
    steps = [W.draw_step_inputs(spec, 0), W.draw_step_inputs(spec, 1)]
    ref_cs, ref_state = x.conv_state.copy(), x.state.copy()   # the oracle's own pools
    for step, st in enumerate(steps):
        if step == 1:  # new token inputs, same pools: the state carries over
            for d in (dA, dB):
                d["qkv"].copy_(T.bf16_tensor(st["qkv"], cuda_device))
                d["g"].copy_(torch.from_numpy(st["g"]))
                d["beta"].copy_(T.bf16_tensor(st["beta"], cuda_device))
                d["gate"].copy_(T.bf16_tensor(st["gate"], cuda_device))
        callA(stream)
        rc = _noalloc(callB, stream)
        assert rc == 0, binding.load_library().kda_last_error().decode()
        torch.cuda.synchronize(cuda_device)
        ref = oracle.decode(qkv=st["qkv"], conv_weight=x.conv_weight, conv_state=ref_cs, state=ref_state,
                            g=st["g"], beta=st["beta"], slot_idx=x.slot_idx, H=x.H, gate=st["gate"],
                            norm_weight=x.norm_weight, eps=spec.eps, in_place=True)
        assert int(dA["err_flag"].item()) == 0 and int(dB["err_flag"].item()) == 0
        what = f"call {step + 1}"
        # against the oracle: output, conv state bit-exact, state per slot
        T.check_out(T.bf16_bits(dB["out"]), ref, what)
        assert np.array_equal(T.bf16_bits(dB["conv_state"]), ref_cs), f"{what}: conv state vs oracle"
        sb = dB["state"].cpu().numpy()
        for s in range(spec.num_slots):
            T.check_state_slot(sb[s], ref_state[s], f"{what} slot {s} vs oracle")
        # against kda_decode on the same inputs
        a = W.bf16_bits_to_f32(T.bf16_bits(dA["out"])).astype(np.float64)
        b = W.bf16_bits_to_f32(T.bf16_bits(dB["out"])).astype(np.float64)
        assert np.abs(a - b).max() <= T.OUT_ATOL, f"{what}: output differs from kda_decode"
        assert np.array_equal(T.bf16_bits(dA["conv_state"]), T.bf16_bits(dB["conv_state"])), \
            f"{what}: conv state differs from kda_decode"
        sa = dA["state"].cpu().numpy()
        for s in range(spec.num_slots):
            T.check_state_slot(sb[s], sa[s], f"{what} slot {s} vs kda_decode")
