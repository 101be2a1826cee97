"""GPU parity of the chunked prefill (``kda_prefill``) against the fp64
prefill oracle (the decode recurrence run token by token).

Tolerances are the decode step's: bf16 output within 3e-2 and within one
bf16 ulp (+1e-5) of the exact value; recurrent state within 1e-4 + 1e-4|ref|
(fp32 arithmetic; the tensor-core products use split tf32 operands, whose
three partial products keep about 21 significant bits per operand); conv
state bit-exact; every slot no sequence uses bit-identical.
"""
import numpy as np
import pytest
import torch

import kda_testlib as T
import oracle
from linear_attention_decode_04_gb300 import KdaPrefillCall, kda_decode, kda_prefill
from linear_attention_decode_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def to_device(x: W.PrefillInputs, dev, out_row_pad: int = 0):
    D = x.spec.H * W.HEAD_DIM
    d = dict(
        qkv=T.bf16_tensor(x.qkv, dev), conv_weight=torch.from_numpy(x.conv_weight).to(dev),
        conv_bias=None if x.conv_bias is None else torch.from_numpy(x.conv_bias).to(dev),
        conv_state=T.bf16_tensor(x.conv_state, dev), state=torch.from_numpy(x.state).to(dev),
        g=torch.from_numpy(x.g).to(dev), beta=T.bf16_tensor(x.beta, dev),
        gate=T.bf16_tensor(x.gate, dev), norm_weight=torch.from_numpy(x.norm_weight).to(dev),
        cu_seqlens=torch.from_numpy(x.cu_seqlens).to(dev), cu_seqlens_cpu=torch.from_numpy(x.cu_seqlens),
        slot_idx=torch.from_numpy(x.slot_idx).to(dev),
        err_flag=torch.zeros(1, dtype=torch.int32, device=dev))
    # NaN-filled: any row the kernel should write and does not is caught
    d["out_full"] = torch.full((x.spec.T, D + out_row_pad), float("nan"), dtype=torch.bfloat16, device=dev)
    d["out"] = d["out_full"][:, :D]
    return d


def run_gpu(x: W.PrefillInputs, d: dict):
    kda_prefill(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                d["cu_seqlens"], d["slot_idx"], d["out"], cu_seqlens_cpu=d["cu_seqlens_cpu"], gate=d["gate"],
                norm_weight=d["norm_weight"], conv_bias=d["conv_bias"], eps=x.spec.eps,
                out_norm=x.spec.out_norm, err_flag=d["err_flag"])


def run_oracle(x: W.PrefillInputs, seqs=None):
    """Oracle over all sequences, or over a subset (sequences are independent:
    the subset is re-batched with its own cu_seqlens)."""
    if seqs is None:
        return oracle.prefill(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state,
                              g=x.g, beta=x.beta, gate=x.gate, norm_weight=x.norm_weight,
                              conv_bias=x.conv_bias, slot_idx=x.slot_idx, cu_seqlens=x.cu_seqlens,
                              H=x.spec.H, eps=x.spec.eps, out_norm=x.spec.out_norm), None
    rows = np.concatenate([np.arange(x.cu_seqlens[b], x.cu_seqlens[b + 1]) for b in seqs]).astype(np.int64)
    lens = [int(x.cu_seqlens[b + 1] - x.cu_seqlens[b]) for b in seqs]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    r = oracle.prefill(qkv=x.qkv[rows], conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state,
                       g=x.g[rows], beta=x.beta[rows], gate=x.gate[rows], norm_weight=x.norm_weight,
                       conv_bias=x.conv_bias, slot_idx=x.slot_idx[list(seqs)], cu_seqlens=cu,
                       H=x.spec.H, eps=x.spec.eps, out_norm=x.spec.out_norm)
    return r, rows


def compare(x: W.PrefillInputs, d: dict, ref, rows=None, seqs=None):
    out = T.bf16_bits(d["out"])
    if rows is None:
        covered = np.zeros(x.spec.T, bool)
        for b in range(x.spec.B):
            covered[x.cu_seqlens[b]:x.cu_seqlens[b + 1]] = True
        assert covered.all()
        T.check_out(out, ref)
    else:
        T.check_out(out[rows], ref)
    followed = range(x.spec.B) if seqs is None else seqs
    written = {int(x.slot_idx[b]) for b in followed
               if 0 < x.slot_idx[b] < x.spec.num_slots and x.cu_seqlens[b + 1] > x.cu_seqlens[b]}
    used = {int(v) for v in x.slot_idx}
    st = d["state"].cpu().numpy()
    cs = T.bf16_bits(d["conv_state"])
    worst = 0.0
    for s in range(x.spec.num_slots):
        if s in written:
            worst = max(worst, T.check_state_slot(st[s], ref.state[s], f"slot {s}"))
            assert np.array_equal(cs[s], ref.conv_state[s]), f"conv state of slot {s}"
        elif seqs is None or s not in used:
            # no sequence writes it (or the oracle followed every sequence)
            assert np.array_equal(st[s], x.state[s]), f"untouched slot {s} changed"
            assert np.array_equal(cs[s], x.conv_state[s]), f"untouched conv slot {s} changed"
    return worst


@pytest.mark.parametrize("spec", [W.PREFILL_SMALL, W.PREFILL_NORM_OFF, W.PREFILL_STRONG_DECAY],
                         ids=lambda s: s.name)
def test_prefill_matches_oracle(cuda_device, spec):
    x = W.make_prefill_inputs(spec)
    d = to_device(x, cuda_device)
    run_gpu(x, d)
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) == 0
    ref, _ = run_oracle(x)
    compare(x, d, ref)


@pytest.mark.parametrize("sigma,v_scale", [(10.0, 1e-1), (10.0, 1e-2), (30.0, 1e-2), (100.0, 1e-3)])
def test_prefill_cancelling_readout(cuda_device, sigma, v_scale):
    """q~ = k~ exactly (identical conv weights, taps and inputs for the q and
    k channels), beta = 1, g = 0, a state of N(0, sigma) and v conv weights
    scaled by v_scale, over sequences of 37, 70 and 96 tokens: every o_t is
    orders of magnitude below Q_G S0.  The chunk form's plain readout
    Q_G S0 + R Delta lost these outputs (beyond 3e-2 at sigma = 30); the
    rearranged one must keep them within one bf16 ulp.  The state is held to
    its tolerance at sigma = 10 (500 times the workload's state); at 30 and
    100 the absolute floor of the state tolerance scales with sigma / 10, the
    precision of the split tf32 products on states of that size."""
    spec = W.PrefillSpec(f"prefill_cancel_s{sigma:g}_v{v_scale:g}", lens=(37, 70, 96), H=4, num_slots=6, seed=60)
    x = W.make_prefill_inputs(spec)
    D = spec.H * W.HEAD_DIM
    x.conv_weight[1] = x.conv_weight[0]
    x.conv_weight[2] *= np.float32(v_scale)
    x.qkv[:, D:2 * D] = x.qkv[:, 0:D]
    x.conv_state[:, D:2 * D, :] = x.conv_state[:, 0:D, :]
    x.beta[:] = W.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    x.g[:] = 0.0
    x.state *= np.float32(sigma / 0.02)
    d = to_device(x, cuda_device)
    run_gpu(x, d)
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) == 0
    ref, _ = run_oracle(x)
    if sigma <= 10.0:
        compare(x, d, ref)
        return
    T.check_out(T.bf16_bits(d["out"]), ref)
    st, cs = d["state"].cpu().numpy().astype(np.float64), T.bf16_bits(d["conv_state"])
    assert np.array_equal(cs, ref.conv_state), "conv state not bit-exact"
    want = ref.state.astype(np.float64)
    assert np.all(np.abs(st - want) <= T.STATE_ATOL * sigma / 10.0 + T.STATE_RTOL * np.abs(want)), \
        "state beyond 1e-4 (sigma / 10) + 1e-4 |ref|"


def test_prefill_padding_rows_zero_and_row_stride(cuda_device):
    # a padding sequence writes zeros; rows are strided (out row padding untouched)
    x = W.make_prefill_inputs(W.PREFILL_SMALL)
    d = to_device(x, cuda_device, out_row_pad=8)
    run_gpu(x, d)
    torch.cuda.synchronize(cuda_device)
    pad = 4
    rows = slice(int(x.cu_seqlens[pad]), int(x.cu_seqlens[pad + 1]))
    assert np.all(T.bf16_bits(d["out"])[rows] == 0)
    assert torch.isnan(d["out_full"][:, -8:].float()).all()


def test_prefill_full_batch_sampled(cuda_device):
    # the measured batch (16 sequences, 16,384 tokens, H = 48); the oracle
    # follows six sequences: one token, a partial chunk, exact chunks, long
    x = W.make_prefill_inputs(W.PREFILL_BENCH)
    d = to_device(x, cuda_device)
    run_gpu(x, d)
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) == 0
    seqs = (1, 4, 7, 11, 12, 3)
    ref, rows = run_oracle(x, seqs)
    compare(x, d, ref, rows=rows, seqs=seqs)


def test_prefill_then_decode_continues_the_state(cuda_device):
    # prefill a batch, then one decode step on the same pools: both against
    # the oracle chained the same way
    x = W.make_prefill_inputs(W.PREFILL_SMALL)
    d = to_device(x, cuda_device)
    run_gpu(x, d)
    ref, _ = run_oracle(x)
    # one decode token per sequence, same slots
    B, H = x.spec.B, x.spec.H
    step = W.draw_step_inputs(W.Spec("prefill_next_token", N=B, H=H, num_slots=x.spec.num_slots, seed=77))
    out = torch.full((B, H * 128), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    kda_decode(T.bf16_tensor(step["qkv"], cuda_device), d["conv_weight"], d["conv_state"], d["state"],
               torch.from_numpy(step["g"]).to(cuda_device), T.bf16_tensor(step["beta"], cuda_device),
               d["slot_idx"], out, gate=T.bf16_tensor(step["gate"], cuda_device),
               norm_weight=d["norm_weight"], conv_bias=d["conv_bias"], eps=x.spec.eps)
    torch.cuda.synchronize(cuda_device)
    dec = oracle.decode(qkv=step["qkv"], conv_weight=x.conv_weight, conv_state=ref.conv_state,
                        state=ref.state, g=step["g"], beta=step["beta"], slot_idx=x.slot_idx, H=H,
                        gate=step["gate"], norm_weight=x.norm_weight, conv_bias=x.conv_bias, eps=x.spec.eps)
    T.check_out(T.bf16_bits(out), dec)
    st = d["state"].cpu().numpy()
    for s in {int(v) for v in x.slot_idx if v > 0}:
        T.check_state_slot(st[s], dec.state[s], f"slot {s} after prefill + decode")


def test_prefill_device_errors_flagged(cuda_device):
    # a slot past the pool and a decreasing cu_seqlens entry: flagged, the
    # other sequences still correct, nothing written for the bad ones
    x = W.make_prefill_inputs(W.PREFILL_SMALL)
    x.slot_idx[0] = x.spec.num_slots + 3
    d = to_device(x, cuda_device)
    run_gpu(x, d)
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) & 1
    ref, _ = run_oracle(x)
    compare(x, d, ref)

    y = W.make_prefill_inputs(W.PREFILL_SMALL)
    d2 = to_device(y, cuda_device)
    bad = d2["cu_seqlens"].clone()
    bad[2] = bad[1] - 1   # sequence 1 ends before it starts; sequence 2 starts past its end
    d2["cu_seqlens"] = bad
    run_gpu(y, d2)
    torch.cuda.synchronize(cuda_device)
    assert int(d2["err_flag"].item()) & 4


def test_prefill_graph_capture_and_prepared_call(cuda_device):
    x = W.make_prefill_inputs(W.PREFILL_NORM_OFF)
    d = to_device(x, cuda_device)
    call = KdaPrefillCall(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                          d["cu_seqlens"], d["slot_idx"], d["out"], cu_seqlens_cpu=d["cu_seqlens_cpu"],
                          gate=d["gate"], norm_weight=d["norm_weight"], conv_bias=d["conv_bias"],
                          eps=x.spec.eps, out_norm=x.spec.out_norm, err_flag=d["err_flag"])
    state0, cs0 = d["state"].clone(), d["conv_state"].clone()
    s = torch.cuda.Stream(cuda_device)
    call(s)          # eager once (device set-up), then restore the pools and capture
    torch.cuda.synchronize(cuda_device)
    d["state"].copy_(state0)
    d["conv_state"].copy_(cs0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call(s)
    graph.replay()
    torch.cuda.synchronize(cuda_device)
    ref, _ = run_oracle(x)
    compare(x, d, ref)


def test_prefill_long_single_sequence(cuda_device):
    # one sequence of 4,133 tokens (130 chunks, a ragged last one): the state
    # runs through 129 chunk updates before the last outputs
    spec = W.PrefillSpec("prefill_b1_t4133_h4", lens=(4133,), H=4, num_slots=3, seed=61)
    x = W.make_prefill_inputs(spec)
    d = to_device(x, cuda_device)
    run_gpu(x, d)
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) == 0
    ref, _ = run_oracle(x)
    compare(x, d, ref)


def test_prefill_many_short_sequences_and_wide_heads(cuda_device):
    rng = np.random.default_rng(5)
    lens = tuple(int(v) for v in rng.integers(0, 41, 48))  # 0..40 tokens, empty ones included
    for spec in (W.PrefillSpec("prefill_b48_short_h2", lens=lens, H=2, num_slots=64, seed=62,
                               pad_seqs=(3, 17)),
                 W.PrefillSpec("prefill_b3_h96", lens=(33, 64, 7), H=96, num_slots=4, seed=63)):
        x = W.make_prefill_inputs(spec)
        d = to_device(x, cuda_device)
        run_gpu(x, d)
        torch.cuda.synchronize(cuda_device)
        assert int(d["err_flag"].item()) == 0
        ref, _ = run_oracle(x)
        compare(x, d, ref)


def test_prefill_continues_across_calls_strided_qkv_q_scale(cuda_device):
    # a batch prefilled in two calls (first 45 tokens, then the rest of each
    # sequence) equals one call over the whole sequences; qkv rows strided;
    # q_scale given
    spec = W.PrefillSpec("prefill_b2_h2_split", lens=(100, 77), H=2, num_slots=4, seed=64)
    x = W.make_prefill_inputs(spec)
    q_scale = 0.25
    ref = oracle.prefill(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state,
                         g=x.g, beta=x.beta, gate=x.gate, norm_weight=x.norm_weight, slot_idx=x.slot_idx,
                         cu_seqlens=x.cu_seqlens, H=spec.H, eps=spec.eps, q_scale=q_scale)
    dev = cuda_device
    D = spec.H * 128
    qkv_pad = np.zeros((spec.T, 3 * D + 16), np.uint16)
    qkv_pad[:, :3 * D] = x.qkv
    qkv_t = T.bf16_tensor(qkv_pad, dev)
    cs, st = T.bf16_tensor(x.conv_state, dev), torch.from_numpy(x.state).to(dev)
    out = torch.full((spec.T, D), float("nan"), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cw, nw = torch.from_numpy(x.conv_weight).to(dev), torch.from_numpy(x.norm_weight).to(dev)
    g_t, beta_t, gate_t = torch.from_numpy(x.g).to(dev), T.bf16_tensor(x.beta, dev), T.bf16_tensor(x.gate, dev)
    slots = torch.from_numpy(x.slot_idx).to(dev)
    first, second = [], []
    for b in range(spec.B):
        r0, r1 = int(x.cu_seqlens[b]), int(x.cu_seqlens[b + 1])
        first.append(np.arange(r0, r0 + 45))
        second.append(np.arange(r0 + 45, r1))
    for part in (first, second):
        rows = torch.from_numpy(np.concatenate(part)).to(dev)
        cu = np.concatenate([[0], np.cumsum([len(r) for r in part])]).astype(np.int32)
        o_part = torch.empty(len(rows), D, dtype=torch.bfloat16, device=dev)
        kda_prefill(qkv_t[rows][:, :3 * D + 16][:, :], cw, cs, st, g_t[rows].contiguous(),
                    beta_t[rows].contiguous(), torch.from_numpy(cu).to(dev), slots, o_part[:, :],
                    cu_seqlens_cpu=torch.from_numpy(cu), gate=gate_t[rows], norm_weight=nw, eps=spec.eps,
                    q_scale=q_scale, err_flag=err)
        out[rows] = o_part
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0
    T.check_out(T.bf16_bits(out), ref)
    assert np.array_equal(T.bf16_bits(cs), ref.conv_state)
    s_got = st.cpu().numpy()
    for s in {int(v) for v in x.slot_idx}:
        T.check_state_slot(s_got[s], ref.state[s], f"slot {s}")


@pytest.mark.parametrize("lower_bound,with_dt", [(-5.0, True), (0.0, True), (0.0, False)])
def test_prefill_fused_gate(cuda_device, lower_bound, with_dt):
    # KDA_FUSED_GATE: g and beta arrive as raw logits and the chunk kernel
    # activates them (the page's prefill kernel is the fused-gate variant)
    spec = W.PrefillSpec("prefill_gate_b3_h4", lens=(40, 1, 97), H=4, num_slots=6, seed=71, pad_seqs=())
    x = W.make_prefill_inputs(spec)
    rng = np.random.default_rng(72)
    x.g = rng.standard_normal(x.g.shape).astype(np.float32)
    x.beta = W.f32_to_bf16_bits(rng.standard_normal(x.beta.shape).astype(np.float32))
    A_log = (0.5 * rng.standard_normal(spec.H)).astype(np.float32)
    dt_bias = (0.5 * rng.standard_normal(spec.H * 128)).astype(np.float32) if with_dt else None
    d = to_device(x, cuda_device)
    kda_prefill(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"], d["cu_seqlens"],
                d["slot_idx"], d["out"], cu_seqlens_cpu=d["cu_seqlens_cpu"], gate=d["gate"],
                norm_weight=d["norm_weight"], conv_bias=d["conv_bias"], eps=spec.eps, err_flag=d["err_flag"],
                A_log=torch.from_numpy(A_log).to(cuda_device),
                dt_bias=None if dt_bias is None else torch.from_numpy(dt_bias).to(cuda_device),
                lower_bound=lower_bound)
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) == 0
    ref = oracle.prefill(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state, g=x.g,
                         beta=x.beta, gate=x.gate, norm_weight=x.norm_weight, conv_bias=x.conv_bias,
                         slot_idx=x.slot_idx, cu_seqlens=x.cu_seqlens, H=spec.H, eps=spec.eps, fused_gate=True,
                         A_log=A_log, dt_bias=dt_bias, lower_bound=lower_bound)
    compare(x, d, ref)


def test_prefill_sd_conv_state_layout(cuda_device):
    # KDA_CONV_STATE_SD: the conv pool stored tap-first [slots, 3, C]; the
    # whole pool must match the oracle's SD-layout prefill bit for bit
    x = W.make_prefill_inputs(W.PREFILL_SMALL)
    x.conv_state = np.ascontiguousarray(x.conv_state.transpose(0, 2, 1))
    d = to_device(x, cuda_device)
    kda_prefill(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"], d["cu_seqlens"],
                d["slot_idx"], d["out"], cu_seqlens_cpu=d["cu_seqlens_cpu"], gate=d["gate"],
                norm_weight=d["norm_weight"], conv_bias=d["conv_bias"], eps=x.spec.eps, err_flag=d["err_flag"],
                conv_state_layout="SD")
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) == 0
    ref = oracle.prefill(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=x.conv_state, state=x.state, g=x.g,
                         beta=x.beta, gate=x.gate, norm_weight=x.norm_weight, conv_bias=x.conv_bias,
                         slot_idx=x.slot_idx, cu_seqlens=x.cu_seqlens, H=x.spec.H, eps=x.spec.eps,
                         conv_state_sd=True)
    T.check_out(T.bf16_bits(d["out"]), ref)
    assert np.array_equal(T.bf16_bits(d["conv_state"]), ref.conv_state)
    st = d["state"].cpu().numpy()
    for s in range(x.spec.num_slots):
        T.check_state_slot(st[s], ref.state[s], f"slot {s}")


def _prepared(x: W.PrefillInputs, d: dict, **kw):
    return KdaPrefillCall(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                          d["cu_seqlens"], d["slot_idx"], d["out"], cu_seqlens_cpu=d["cu_seqlens_cpu"],
                          gate=d["gate"], norm_weight=d["norm_weight"], conv_bias=d["conv_bias"],
                          eps=x.spec.eps, out_norm=x.spec.out_norm, err_flag=d["err_flag"], **kw)


def _set_order(call, order):
    call.seq_order = order
    call.args.seq_order = order.data_ptr()


def test_prefill_scan_order_changes_nothing(cuda_device):
    # the order in which the scan takes the sequences is a scheduling choice:
    # longest first, index order and reversed give bit-identical results
    x = W.make_prefill_inputs(W.PREFILL_SMALL)
    B = x.spec.B
    got = []
    for order in ("longest", "index", "reversed"):
        d = to_device(x, cuda_device)
        call = _prepared(x, d, longest_first=(order == "longest"))
        assert (call.seq_order is None) == (order != "longest")
        if order == "reversed":
            _set_order(call, torch.arange(B - 1, -1, -1, dtype=torch.int32, device=cuda_device))
        call()
        torch.cuda.synchronize(cuda_device)
        assert int(d["err_flag"].item()) == 0
        got.append((T.bf16_bits(d["out"]), d["state"].cpu().numpy(), T.bf16_bits(d["conv_state"])))
        if order == "longest":
            ref, _ = run_oracle(x)
            compare(x, d, ref)
    for other in got[1:]:
        for a, b in zip(got[0], other):
            assert np.array_equal(a, b)


def test_prefill_scan_order_out_of_range_flagged(cuda_device):
    # an entry outside [0, B) is flagged; the sequence it displaced is left
    # untouched (rows unwritten, pools unchanged) and every other one is right
    x = W.make_prefill_inputs(W.PREFILL_SMALL)
    B, victim = x.spec.B, 3
    assert x.cu_seqlens[victim + 1] > x.cu_seqlens[victim] and x.slot_idx[victim] > 0
    d = to_device(x, cuda_device)
    call = _prepared(x, d, longest_first=False)
    order = torch.arange(B, dtype=torch.int32, device=cuda_device)
    order[victim] = B
    _set_order(call, order)
    call()
    torch.cuda.synchronize(cuda_device)
    assert int(d["err_flag"].item()) & 16
    others = [b for b in range(B) if b != victim]
    ref, rows = run_oracle(x, seqs=others)
    compare(x, d, ref, rows=rows, seqs=others)
    r0, r1 = int(x.cu_seqlens[victim]), int(x.cu_seqlens[victim + 1])
    assert torch.isnan(d["out"][r0:r1].float()).all()
    s = int(x.slot_idx[victim])
    assert np.array_equal(d["state"][s].cpu().numpy(), x.state[s])
    assert np.array_equal(T.bf16_bits(d["conv_state"])[s], x.conv_state[s])
