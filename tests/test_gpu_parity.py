"""CUDA path vs the fp64 oracle on the same seeded inputs, through the C ABI.

Tolerances: conv state and untouched slots bit-exact; recurrent state
|d| <= 1e-4 + 1e-4|ref|; bf16 output |d| <= 3e-2 and, tighter, within one
bf16 ulp of the exact output."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import kda_testlib as T
from linear_attention_decode_04_gb300 import KdaError, kda_decode
from linear_attention_decode_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check(x, dev, early_prefetch=False, queue=False, **kw):
    d = T.to_device(x, dev)
    wq = torch.zeros(2, dtype=torch.int32, device=dev) if queue else None
    T.run_gpu(x, d, early_prefetch=early_prefetch, work_queue=wq, **kw)
    torch.cuda.synchronize()
    ref = T.run_oracle(x, **kw)
    res = T.compare_all(x, d, ref, init_state=x.state, init_conv=x.conv_state)
    assert int(d["err_flag"].item()) == 0
    if queue:
        assert wq.tolist() == [0, 0], "work queue not returned to zero"
    return res


@pytest.mark.parametrize("name", list(W.SPECS))
def test_workload_parity(name, cuda_device):
    """The four seeded workloads of the decode step, compared element by element."""
    x = W.make_inputs(W.SPECS[name])
    res = _check(x, cuda_device)
    print(name, res)


@pytest.mark.parametrize("out_norm", [True, False])
@pytest.mark.parametrize("update_conv_state", [True, False])
def test_flag_combinations(out_norm, update_conv_state, cuda_device):
    x = W.make_inputs(W.Spec("flags_n9_h12_pool16", N=9, H=12, num_slots=16, seed=21, pad_tail=2))
    _check(x, cuda_device, out_norm=out_norm, update_conv_state=update_conv_state)


@pytest.mark.parametrize("name", list(W.SPECS))
@pytest.mark.parametrize("queue", [False, True])
def test_workload_parity_early_prefetch(name, queue, cuda_device):
    """Same results with KDA_EARLY_PREFETCH (state streamed before the
    previous kernel on the stream completes; nothing before it writes the
    pools here), with the static and the work-queue schedule; the queue is
    zero again afterwards."""
    _check(W.make_inputs(W.SPECS[name]), cuda_device, early_prefetch=True, queue=queue)


@pytest.mark.parametrize("name", list(W.SPECS))
def test_workload_parity_work_queue(name, cuda_device):
    _check(W.make_inputs(W.SPECS[name]), cuda_device, queue=True)


def test_back_to_back_same_pool_in_one_graph(cuda_device):
    """Three decode steps on the SAME pools, captured in one CUDA graph
    (programmatic dependent launches, no early prefetch): each step must see
    the previous step's state and conv state, as three oracle steps do."""
    from linear_attention_decode_04_gb300.stack import warm_up
    from linear_attention_decode_04_gb300 import KdaDecodeCall
    spec = W.Spec("chain_n24_h24_pool32", N=24, H=24, num_slots=32, seed=41, pad_tail=3)
    x = W.make_inputs(spec)
    d = T.to_device(x, cuda_device)
    steps = [W.draw_step_inputs(spec, v) for v in range(3)]
    dev_steps, calls = [], []
    queue = torch.zeros(2, dtype=torch.int32, device=cuda_device)
    for st in steps:
        ds = dict(qkv=T.bf16_tensor(st["qkv"], cuda_device), g=torch.from_numpy(st["g"]).to(cuda_device),
                  beta=T.bf16_tensor(st["beta"], cuda_device), gate=T.bf16_tensor(st["gate"], cuda_device),
                  out=torch.empty(x.N, x.H * 128, dtype=torch.bfloat16, device=cuda_device))
        dev_steps.append(ds)
        calls.append(KdaDecodeCall(ds["qkv"], d["conv_weight"], d["conv_state"], d["state"], ds["g"],
                                   ds["beta"], d["slot_idx"], ds["out"], gate=ds["gate"],
                                   norm_weight=d["norm_weight"], eps=spec.eps, err_flag=d["err_flag"],
                                   work_queue=queue))
    warm_up(cuda_device)
    s = torch.cuda.Stream(cuda_device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    cs, stt = x.conv_state.copy(), x.state.copy()
    import oracle
    for st, ds in zip(steps, dev_steps):
        ref = oracle.decode(qkv=st["qkv"], conv_weight=x.conv_weight, conv_state=cs, state=stt, g=st["g"],
                            beta=st["beta"], slot_idx=x.slot_idx, H=x.H, gate=st["gate"],
                            norm_weight=x.norm_weight, eps=spec.eps, in_place=True)
        T.check_out(T.bf16_bits(ds["out"]), ref, "chained step")
    assert np.array_equal(T.bf16_bits(d["conv_state"]), cs)
    for sl in range(spec.num_slots):
        T.check_state_slot(d["state"][sl].cpu().numpy(), stt[sl], f"slot {sl}")
    assert int(d["err_flag"].item()) == 0
    assert queue.tolist() == [0, 0]


@pytest.mark.parametrize("H", [12, 24, 48, 96, 5])
@pytest.mark.parametrize("N", [1, 7])
def test_heads_and_rows(H, N, cuda_device):
    """Every supported head count (12/24/48/96 = 96 heads over TP 8/4/2/1),
    an unusual one, and the odd row count 7."""
    x = W.make_inputs(W.Spec(f"h{H}_n{N}", N=N, H=H, num_slots=N + 3, seed=100 + H + N))
    _check(x, cuda_device)


def test_negative_and_zero_slots_are_padding(cuda_device):
    spec = W.Spec("pad_mix_n6_h12", N=6, H=12, num_slots=8, seed=31, slots=(0, 4, -3, 7, 0, 2))
    x = W.make_inputs(spec)
    res = _check(x, cuda_device)
    assert res["out_max_abs"] <= T.OUT_ATOL


def test_all_padding_batch(cuda_device):
    x = W.make_inputs(W.Spec("all_pad_n5_h24", N=5, H=24, num_slots=4, seed=32, slots=(0, 0, -1, 0, 0)))
    d = T.to_device(x, cuda_device)
    T.run_gpu(x, d)
    torch.cuda.synchronize()
    assert not torch.any(d["out"].float() != 0)
    assert np.array_equal(d["state"].cpu().numpy(), x.state)
    assert np.array_equal(T.bf16_bits(d["conv_state"]), x.conv_state)


def test_out_of_range_slot_sets_flag_without_trap(cuda_device):
    x = W.make_inputs(W.Spec("oob_n4_h12", N=4, H=12, num_slots=6, seed=33, slots=(1, 6, 3, 1000)))
    d = T.to_device(x, cuda_device)
    T.run_gpu(x, d)
    torch.cuda.synchronize()
    assert int(d["err_flag"].item()) == 1
    ref = T.run_oracle(x)
    assert ref.n_out_of_range == 2
    T.compare_all(x, d, ref, init_state=x.state, init_conv=x.conv_state)


def test_bias_and_row_strides(cuda_device):
    """Conv bias, a qkv row longer than 3*H*128, and row-strided gate/out
    views; the padding columns of out stay unwritten."""
    spec = W.Spec("strided_n5_h12", N=5, H=12, num_slots=9, seed=34, with_bias=True, qkv_row_pad=24,
                  pad_tail=1)
    x = W.make_inputs(spec)
    d = T.to_device(x, cuda_device, out_row_pad=16, gate_row_pad=8)
    T.run_gpu(x, d)
    torch.cuda.synchronize()
    ref = T.run_oracle(x)
    T.compare_all(x, d, ref, init_state=x.state, init_conv=x.conv_state)
    assert torch.isnan(d["out_full"][:, x.H * 128:].float()).all()


def test_q_scale_argument(cuda_device):
    x = W.make_inputs(replace(W.NORM_OFF, name="qscale_n16_h12", N=16, H=12, num_slots=20))
    _check(x, cuda_device, q_scale=1.0)


def test_deterministic_repeat(cuda_device):
    x = W.make_inputs(W.PAD_TAIL)
    outs = []
    for _ in range(2):
        d = T.to_device(x, cuda_device)
        T.run_gpu(x, d)
        torch.cuda.synchronize()
        outs.append((T.bf16_bits(d["out"]), d["state"].cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_pool_guard_regions_untouched(cuda_device):
    """Allocate the pools with guard slots on both sides (sentinel-filled) and
    pass the middle: nothing outside the passed pool is written."""
    x = W.make_inputs(W.Spec("guard_n8_h12", N=8, H=12, num_slots=10, seed=35, pad_tail=1))
    d = T.to_device(x, cuda_device)
    S, H, C = x.spec.num_slots, x.H, x.C
    big = torch.full((S + 2, H, 128, 128), 7.25, dtype=torch.float32, device=cuda_device)
    big[1:S + 1] = d["state"]
    bigcs = torch.full((S + 2, C, 3), -2.0, dtype=torch.bfloat16, device=cuda_device)
    bigcs[1:S + 1] = d["conv_state"]
    d["state"], d["conv_state"] = big[1:S + 1], bigcs[1:S + 1]
    T.run_gpu(x, d)
    torch.cuda.synchronize()
    assert torch.all(big[0] == 7.25) and torch.all(big[S + 1] == 7.25)
    assert torch.all(bigcs[0] == -2.0) and torch.all(bigcs[S + 1] == -2.0)
    T.compare_all(x, d, T.run_oracle(x))


def test_binding_rejects_cpu_and_bad_shapes(cuda_device):
    x = W.make_inputs(W.PR1_REF)
    d = T.to_device(x, cuda_device)
    with pytest.raises(ValueError):
        kda_decode(d["qkv"].cpu(), d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                   d["slot_idx"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"])
    with pytest.raises(ValueError):
        kda_decode(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"][:, :5], d["beta"],
                   d["slot_idx"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"])
    # misaligned qkv (offset by one element) is refused by the C ABI itself
    raw = torch.empty(x.N * x.C + 8, dtype=torch.bfloat16, device=cuda_device)
    mis = raw[1:1 + x.N * x.C].view(x.N, x.C)
    with pytest.raises(KdaError) as ei:
        kda_decode(mis, d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                   d["slot_idx"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"])
    assert ei.value.status == -3


@pytest.mark.parametrize("early_prefetch", [False, True])
@pytest.mark.parametrize("queue", [False, True])
def test_bounded_wait_runs_out_and_reports(early_prefetch, queue, cuda_device):
    """Failure path without a GPU fault: one unit's load is never signalled
    and the waits are limited to 20 ms.  The launch must return (no hang, no
    trap) with KDA_DEVERR_TIMEOUT set, and the context must stay usable: a
    normal call afterwards still matches the oracle."""
    from linear_attention_decode_04_gb300 import KdaDecodeCall
    from linear_attention_decode_04_gb300.binding import KDA_DEVERR_TIMEOUT
    x = W.make_inputs(W.Spec("waittest_n40_h24_pool48", N=40, H=24, num_slots=48, seed=51, pad_tail=2))
    d = T.to_device(x, cuda_device)
    wq = torch.zeros(2, dtype=torch.int32, device=cuda_device) if queue else None
    call = KdaDecodeCall(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                         d["slot_idx"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"],
                         eps=x.spec.eps, err_flag=d["err_flag"], early_prefetch=early_prefetch,
                         work_queue=wq)
    # withhold a static unit, or (with the queue) one handed out dynamically
    call.wait_test(20_000_000, withhold_unit=0 if not queue else x.N * x.H - 5)
    torch.cuda.synchronize()
    assert int(d["err_flag"].item()) & KDA_DEVERR_TIMEOUT
    if queue:
        assert wq.tolist() == [0, 0], "work queue not reset after the aborted launch"
    # the context is intact: a fresh problem decodes correctly
    _check(W.make_inputs(W.PAD_TAIL), cuda_device)


@pytest.mark.parametrize("lower_bound", [-5.0, 0.0])
@pytest.mark.parametrize("with_bias", [True, False])
def test_fused_gate_parity(lower_bound, with_bias, cuda_device):
    """KDA_FUSED_GATE: g and beta arrive as raw logits and are activated in
    the kernel (bounded form with lower_bound < 0, softplus form otherwise)."""
    import oracle
    spec = W.Spec("gate_n20_h24_pool32", N=20, H=24, num_slots=32, seed=61, pad_tail=2)
    x = W.make_inputs(spec)
    rng = np.random.default_rng(62)
    x.g = rng.standard_normal(x.g.shape).astype(np.float32)                    # raw gate logits
    x.beta = W.f32_to_bf16_bits(rng.standard_normal(x.beta.shape).astype(np.float32))
    A_log = (0.5 * rng.standard_normal(x.H)).astype(np.float32)
    dt_bias = (0.5 * rng.standard_normal(x.H * 128)).astype(np.float32) if with_bias else None
    d = T.to_device(x, cuda_device)
    kda_decode(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"], d["slot_idx"],
               d["out"], gate=d["gate"], norm_weight=d["norm_weight"], eps=spec.eps, err_flag=d["err_flag"],
               A_log=torch.from_numpy(A_log).to(cuda_device),
               dt_bias=None if dt_bias is None else torch.from_numpy(dt_bias).to(cuda_device),
               lower_bound=lower_bound)
    torch.cuda.synchronize()
    ref = oracle.decode(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state, g=x.g,
                        beta=x.beta, slot_idx=x.slot_idx, H=x.H, gate=x.gate, norm_weight=x.norm_weight,
                        eps=spec.eps, fused_gate=True, A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound)
    T.compare_all(x, d, ref, init_state=x.state, init_conv=x.conv_state)
    assert int(d["err_flag"].item()) == 0


@pytest.mark.parametrize("name", ["n4_h12_pool8", "n32_h24_pool64_pad8", "n128_h48_pool512_normoff"])
@pytest.mark.parametrize("update_conv_state", [True, False])
def test_sd_conv_state_layout(name, update_conv_state, cuda_device):
    """KDA_CONV_STATE_SD: the conv state stored tap-first [slots, 3, C]; the
    whole pool must match the oracle's SD-layout step bit for bit."""
    import oracle
    x = W.make_inputs(W.SPECS[name])
    cs_sd = np.ascontiguousarray(x.conv_state.transpose(0, 2, 1))
    d = T.to_device(x, cuda_device)
    d["conv_state"] = T.bf16_tensor(cs_sd, cuda_device)
    kda_decode(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"], d["slot_idx"],
               d["out"], gate=d["gate"], norm_weight=d["norm_weight"], eps=x.spec.eps, err_flag=d["err_flag"],
               out_norm=x.spec.out_norm, update_conv_state=update_conv_state, conv_state_layout="SD")
    torch.cuda.synchronize()
    ref = oracle.decode(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=cs_sd, state=x.state, g=x.g,
                        beta=x.beta, slot_idx=x.slot_idx, H=x.H, gate=x.gate, norm_weight=x.norm_weight,
                        eps=x.spec.eps, out_norm=x.spec.out_norm, update_conv_state=update_conv_state,
                        conv_state_sd=True)
    T.check_out(T.bf16_bits(d["out"]), ref)
    assert np.array_equal(T.bf16_bits(d["conv_state"]), ref.conv_state), "SD conv state not bit-exact"
    for s in range(x.spec.num_slots):
        T.check_state_slot(d["state"][s].cpu().numpy(), ref.state[s], f"slot {s}")
    assert int(d["err_flag"].item()) == 0


@pytest.mark.parametrize("sigma,v_scale,out_norm", [(10.0, 1e-2, True), (100.0, 1e-1, True),
                                                     (30.0, 3e-3, True), (30.0, 3e-3, False)])
def test_cancelling_readout(sigma, v_scale, out_norm, cuda_device):
    """q~ = k~ exactly, beta = 1, g = 0, a state of N(0, sigma) and a small v:
    the readout o is orders of magnitude below A^T q^, so an fp32 readout or
    RMSNorm sum that cancels late loses the output (the CPU emulation in
    test_readout_cancellation.py shows the earlier expansion of sum o^2
    missing 3e-2 on these inputs).  Output within 3e-2 and one bf16 ulp of the
    exact value, state within its tolerance, conv state bit-exact."""
    x = T.cancellation_inputs(sigma, v_scale, N=24, H=12, out_norm=out_norm)
    _check(x, cuda_device)
    _check(x, cuda_device, queue=True)
