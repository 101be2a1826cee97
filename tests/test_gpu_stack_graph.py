"""The 69-layer decode step as one CUDA graph, replayed 100 times with state
carried across steps, checked against the oracle after steps 1, 10 and 100.

Every layer has its own weights, conv state and 96-slot state pool (H=48,
N=64 rows, the last 4 slot-0 padding).  Each step feeds one of four seeded
per-token input draws (copied into the graph's static input buffers before
the replay).  The oracle follows one whole layer (every row, every slot,
untouched slots bit-exact) and a sample of rows of three more layers.
"""
import numpy as np
import pytest
import torch

import kda_testlib as T
import oracle
from linear_attention_decode_04_gb300 import workloads as W
from linear_attention_decode_04_gb300.stack import STEP_INPUTS, DecodeStack

pytestmark = pytest.mark.gpu

FULL_LAYER = 68
SAMPLED_LAYERS = (0, 1, 34)
SAMPLED_ROWS = np.array([0, 7, 23, 41, 59, 60, 63])  # 60..63 are padding rows
VARIANTS = 4
CHECK_AT = (1, 10, 100)


def _dev_step(var, device):
    return dict(qkv=T.bf16_tensor(var["qkv"], device), g=torch.from_numpy(var["g"]).to(device),
                beta=T.bf16_tensor(var["beta"], device), gate=T.bf16_tensor(var["gate"], device))


def test_stack69_graph_replay_carries_state(cuda_device):
    dev = cuda_device
    layers, host = [], {}
    for ell in range(W.STACK_LAYERS):
        x = W.make_inputs(W.stack_layer_spec(ell))
        L = T.to_device(x, dev)
        L["out"] = L["out_full"]
        variants = [W.draw_step_inputs(x.spec, v) for v in range(VARIANTS)]
        L["variants"] = [_dev_step(v, dev) for v in variants]
        layers.append(L)
        if ell == FULL_LAYER or ell in SAMPLED_LAYERS:
            host[ell] = (x, variants)
    spec = W.STACK_LAYER
    stack = DecodeStack(layers, eps=spec.eps, out_norm=spec.out_norm,
                        update_conv_state=spec.update_conv_state)
    stack.capture()
    assert stack.launches_per_step == W.STACK_LAYERS

    for t in range(1, max(CHECK_AT) + 1):
        v = (t - 1) % VARIANTS
        for L in layers:
            for k in STEP_INPUTS:
                if k != "slot_idx":
                    L[k].copy_(L["variants"][v][k])
        stack.replay()
        refs = {}
        for ell, (x, variants) in host.items():
            var = variants[v]
            rows = np.arange(x.N) if ell == FULL_LAYER else SAMPLED_ROWS
            refs[ell] = (rows, oracle.decode(
                qkv=var["qkv"][rows], conv_weight=x.conv_weight, conv_state=x.conv_state,
                state=x.state, g=var["g"][rows], beta=var["beta"][rows], slot_idx=x.slot_idx[rows],
                H=x.H, gate=var["gate"][rows], norm_weight=x.norm_weight, eps=x.spec.eps,
                in_place=True))
        if t not in CHECK_AT:
            continue
        torch.cuda.synchronize(dev)
        for ell, (rows, ref) in refs.items():
            x = host[ell][0]
            L = layers[ell]
            assert int(L["err_flag"].item()) == 0
            T.check_out(T.bf16_bits(L["out"])[rows], ref, f"layer {ell} step {t}")
            slots = [int(s) for s in x.slot_idx[rows] if s > 0]
            st = L["state"]
            cs = T.bf16_bits(L["conv_state"])
            for s in slots:
                T.check_state_slot(st[s].cpu().numpy(), x.state[s], f"layer {ell} step {t} slot {s}")
                assert np.array_equal(cs[s], x.conv_state[s]), f"layer {ell} step {t} conv slot {s}"
            if ell == FULL_LAYER:
                active = set(int(s) for s in x.slot_idx if s > 0)
                init = W.make_inputs(W.stack_layer_spec(ell))
                for s in range(x.spec.num_slots):
                    if s not in active:
                        assert np.array_equal(st[s].cpu().numpy(), init.state[s]), f"untouched slot {s}"
                        assert np.array_equal(cs[s], init.conv_state[s])
