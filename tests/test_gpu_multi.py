"""Multi-token (speculative) decode on the GPU against the fp64 oracle, through
the C ABI.  Sequence n starts from src_slot[n] and runs T = 1 + num_spec
tokens; the state and window after token t go to dst_slots[n, t].

Tolerances as for the decode step: conv state bit-exact over the whole pool,
untouched slots bit-exact, written slots |d| <= 1e-4 + 1e-4|ref|, bf16
output within 3e-2 and within one bf16 ulp of the exact value."""
import numpy as np
import pytest
import torch

import kda_testlib as T
import oracle
from linear_attention_decode_04_gb300 import KdaDecodeCall
from linear_attention_decode_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _dev(x: W.MultiInputs, dev, conv_sd=False):
    cs = np.ascontiguousarray(x.conv_state.transpose(0, 2, 1)) if conv_sd else x.conv_state
    D = x.H * 128
    return dict(
        qkv=T.bf16_tensor(x.qkv, dev), conv_weight=torch.from_numpy(x.conv_weight).to(dev),
        conv_state=T.bf16_tensor(cs, dev), state=torch.from_numpy(x.state).to(dev),
        g=torch.from_numpy(x.g).to(dev), beta=T.bf16_tensor(x.beta, dev), gate=T.bf16_tensor(x.gate, dev),
        norm_weight=torch.from_numpy(x.norm_weight).to(dev),
        src_slot=torch.from_numpy(x.src_slot).to(dev), dst_slots=torch.from_numpy(x.dst_slots).to(dev),
        out=torch.full((x.N * x.T, D), float("nan"), dtype=torch.bfloat16, device=dev),
        err_flag=torch.zeros(1, dtype=torch.int32, device=dev))


def _call(x, d, src=True, queue=None, early=False, conv_sd=False, **kw):
    return KdaDecodeCall(d["qkv"], d["conv_weight"], d["conv_state"], d["state"], d["g"], d["beta"],
                         d["dst_slots"], d["out"], gate=d["gate"], norm_weight=d["norm_weight"],
                         eps=x.spec.eps, out_norm=x.spec.out_norm, update_conv_state=x.spec.update_conv_state,
                         err_flag=d["err_flag"], tokens_per_seq=x.T, src_slot=d["src_slot"] if src else None,
                         work_queue=queue, early_prefetch=early,
                         conv_state_layout="SD" if conv_sd else "DS", **kw)


def _oracle(x, conv_sd=False, **kw):
    cs = np.ascontiguousarray(x.conv_state.transpose(0, 2, 1)) if conv_sd else x.conv_state
    return oracle.decode_multi(qkv=x.qkv, conv_weight=x.conv_weight, conv_state=cs, state=x.state, g=x.g,
                               beta=x.beta, src_slot=x.src_slot, dst_slots=x.dst_slots, H=x.H, gate=x.gate,
                               norm_weight=x.norm_weight, eps=x.spec.eps, out_norm=x.spec.out_norm,
                               update_conv_state=x.spec.update_conv_state, conv_state_sd=conv_sd, **kw)


def _compare(x, d, ref, conv_sd=False, expect_err=0):
    torch.cuda.synchronize()
    T.check_out(T.bf16_bits(d["out"]), ref, "multi-token out")
    assert np.array_equal(T.bf16_bits(d["conv_state"]), ref.conv_state), "conv state not bit-exact"
    written = {int(s) for s in x.dst_slots.ravel() if 0 < s < x.spec.num_slots}
    st = d["state"].cpu().numpy()
    for s in range(x.spec.num_slots):
        if s in written:
            T.check_state_slot(st[s], ref.state[s], f"slot {s}")
        else:
            assert np.array_equal(st[s], x.state[s]), f"untouched slot {s} changed"
    assert int(d["err_flag"].item()) == expect_err


@pytest.mark.parametrize("Tn", [2, 4, 8])
@pytest.mark.parametrize("out_norm", [True, False])
def test_multi_token_parity(Tn, out_norm, cuda_device):
    spec = W.MultiSpec(f"spec_n9_t{Tn}_h24", N=9, T=Tn, H=24, num_slots=9 * (Tn + 1) + 5, seed=310 + Tn,
                       out_norm=out_norm)
    x = W.make_multi_inputs(spec)
    d = _dev(x, cuda_device)
    _call(x, d)()
    _compare(x, d, _oracle(x))


@pytest.mark.parametrize("Tn", [3, 6])
def test_cancelling_readout(Tn, cuda_device):
    """Every token in the regime where the readout cancels: q~ = k~ exactly
    (identical conv weights, taps and inputs for the q and k channels),
    beta = 1, g = 0, a source state of N(0, 30) and v conv weights scaled by
    1e-2.  Each token's o is then orders of magnitude below A^T q^; the
    outputs must still be within one bf16 ulp of the exact value.  T = 3 and
    6 run the kernel built for up to 4 and up to 8 tokens."""
    spec = W.MultiSpec(f"spec_n8_t{Tn}_h12_cancel", N=8, T=Tn, H=12, num_slots=8 * (Tn + 1) + 3, seed=340 + Tn)
    x = W.make_multi_inputs(spec)
    D = x.H * 128
    x.conv_weight[1] = x.conv_weight[0]
    x.conv_weight[2] *= np.float32(1e-2)
    x.qkv[:, D:2 * D] = x.qkv[:, 0:D]
    x.conv_state[:, D:2 * D, :] = x.conv_state[:, 0:D, :]
    x.beta[:] = W.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    x.g[:] = 0.0
    x.state *= np.float32(30.0 / 0.02)
    d = _dev(x, cuda_device)
    _call(x, d)()
    _compare(x, d, _oracle(x))


def test_t1_with_source_slot(cuda_device):
    """T = 1 with a separate source: decode into a fresh slot (copy on write)."""
    x = W.make_multi_inputs(W.MultiSpec("spec_n16_t1_h12", N=16, T=1, H=12, num_slots=40, seed=320))
    d = _dev(x, cuda_device)
    _call(x, d)()
    _compare(x, d, _oracle(x))


def test_source_from_first_destination(cuda_device):
    """Without src_slot each sequence starts from its first destination slot."""
    x = W.make_multi_inputs(W.MultiSpec("spec_n8_t3_h12_nosrc", N=8, T=3, H=12, num_slots=40, seed=321))
    x.src_slot = x.dst_slots[:, 0].copy()
    d = _dev(x, cuda_device)
    _call(x, d, src=False)()
    _compare(x, d, _oracle(x))


def test_absent_tokens_padding_sequences_and_aliasing(cuda_device):
    """Absent tokens (first, middle, last, all), padding sequences, and each
    sequence's last token stored back into its own source slot."""
    spec = W.MultiSpec("spec_n10_t4_h12_mixed", N=10, T=4, H=12, num_slots=60, seed=322,
                       pad_seqs=(3, 9), absent=((0, 1), (1, 0), (2, 3), (4, 0), (4, 1), (4, 2), (4, 3)),
                       alias_last=True)
    x = W.make_multi_inputs(spec)
    d = _dev(x, cuda_device)
    _call(x, d)()
    _compare(x, d, _oracle(x))


def test_out_of_range_slots_raise_the_flag(cuda_device):
    spec = W.MultiSpec("spec_n6_t2_h12_oob", N=6, T=2, H=12, num_slots=20, seed=323)
    x = W.make_multi_inputs(spec)
    x.src_slot[1] = 500          # whole sequence out of range
    x.dst_slots[2, 1] = 20       # one token out of range
    d = _dev(x, cuda_device)
    _call(x, d)()
    ref = _oracle(x)
    assert ref.n_out_of_range == 2
    _compare(x, d, ref, expect_err=1)


@pytest.mark.parametrize("update_conv_state", [True, False])
def test_sd_layout_and_update_flag(update_conv_state, cuda_device):
    spec = W.MultiSpec("spec_n7_t3_h24_sd", N=7, T=3, H=24, num_slots=40, seed=324,
                       update_conv_state=update_conv_state, absent=((3, 1),))
    x = W.make_multi_inputs(spec)
    d = _dev(x, cuda_device, conv_sd=True)
    _call(x, d, conv_sd=True)()
    _compare(x, d, _oracle(x, conv_sd=True))


@pytest.mark.parametrize("queue", [False, True])
@pytest.mark.parametrize("early", [False, True])
def test_schedules(queue, early, cuda_device):
    """Static and work-queue schedules, with and without early prefetch, on a
    batch with more units than SMs (several units per CTA)."""
    spec = W.MultiSpec("spec_n24_t3_h24", N=24, T=3, H=24, num_slots=100, seed=325, pad_seqs=(5,))
    x = W.make_multi_inputs(spec)
    d = _dev(x, cuda_device)
    wq = torch.zeros(2, dtype=torch.int32, device=cuda_device) if queue else None
    _call(x, d, queue=wq, early=early)()
    _compare(x, d, _oracle(x))
    if queue:
        assert wq.tolist() == [0, 0]


def test_fused_gate(cuda_device):
    spec = W.MultiSpec("spec_n6_t3_h12_gate", N=6, T=3, H=12, num_slots=30, seed=326)
    x = W.make_multi_inputs(spec)
    rng = np.random.default_rng(327)
    x.g = rng.standard_normal(x.g.shape).astype(np.float32)
    x.beta = W.f32_to_bf16_bits(rng.standard_normal(x.beta.shape).astype(np.float32))
    A_log = (0.5 * rng.standard_normal(x.H)).astype(np.float32)
    dt_bias = (0.5 * rng.standard_normal(x.H * 128)).astype(np.float32)
    d = _dev(x, cuda_device)
    _call(x, d, A_log=torch.from_numpy(A_log).to(cuda_device),
          dt_bias=torch.from_numpy(dt_bias).to(cuda_device), lower_bound=-5.0)()
    _compare(x, d, _oracle(x, fused_gate=True, A_log=A_log, dt_bias=dt_bias, lower_bound=-5.0))


def test_two_speculative_steps_in_one_graph(cuda_device):
    """Two multi-token steps captured in one CUDA graph: the second starts
    from a slot the first one wrote (the state after the first accepted
    token), as a speculative decoder would after verification."""
    from linear_attention_decode_04_gb300.stack import warm_up
    spec = W.MultiSpec("spec_n12_t3_h12_chain", N=12, T=3, H=12, num_slots=100, seed=328)
    x = W.make_multi_inputs(spec)
    d = _dev(x, cuda_device)
    # step 2: new token inputs, source = step 1's slot after its second token,
    # destinations = fresh slots
    x2 = W.make_multi_inputs(W.MultiSpec("spec_n12_t3_h12_chain2", N=12, T=3, H=12, num_slots=100, seed=329))
    used = set(x.src_slot.tolist()) | set(x.dst_slots.ravel().tolist())
    free = np.array([s for s in range(1, 100) if s not in used], np.int32)
    src2 = x.dst_slots[:, 1].copy()
    dst2 = free[:12 * 3].reshape(12, 3)
    d2 = dict(d)
    for k in ("qkv", "g", "beta", "gate"):
        d2[k] = {"qkv": T.bf16_tensor(x2.qkv, cuda_device), "g": torch.from_numpy(x2.g).to(cuda_device),
                 "beta": T.bf16_tensor(x2.beta, cuda_device), "gate": T.bf16_tensor(x2.gate, cuda_device)}[k]
    d2["src_slot"] = torch.from_numpy(src2).to(cuda_device)
    d2["dst_slots"] = torch.from_numpy(dst2).to(cuda_device)
    d2["out"] = torch.full_like(d["out"], float("nan"))
    c1, c2 = _call(x, d), _call(x, d2)
    warm_up(cuda_device)
    c1()  # once eagerly (library set-up), then on fresh pools inside the graph
    torch.cuda.synchronize()
    d["state"].copy_(torch.from_numpy(x.state))
    d["conv_state"].copy_(T.bf16_tensor(x.conv_state, cuda_device))
    s = torch.cuda.Stream(cuda_device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c1()
        c2()
    g.replay()
    torch.cuda.synchronize()
    r1 = _oracle(x)
    r2 = oracle.decode_multi(qkv=x2.qkv, conv_weight=x.conv_weight, conv_state=r1.conv_state, state=r1.state,
                             g=x2.g, beta=x2.beta, src_slot=src2, dst_slots=dst2, H=x.H, gate=x2.gate,
                             norm_weight=x.norm_weight, eps=spec.eps)
    T.check_out(T.bf16_bits(d["out"]), r1, "step 1")
    T.check_out(T.bf16_bits(d2["out"]), r2, "step 2")
    assert np.array_equal(T.bf16_bits(d["conv_state"]), r2.conv_state)
    st = d["state"].cpu().numpy()
    for sl in set(dst2.ravel().tolist()) | set(x.dst_slots.ravel().tolist()):
        T.check_state_slot(st[sl], r2.state[sl], f"slot {sl}")
    assert int(d["err_flag"].item()) == 0


def test_bounded_wait_runs_out_and_reports(cuda_device):
    """Failure path without a GPU fault, on the multi-token kernel: one
    unit's inputs are never signalled, the waits are limited to 20 ms; the
    launch returns with KDA_DEVERR_TIMEOUT and the context stays usable."""
    from linear_attention_decode_04_gb300.binding import KDA_DEVERR_TIMEOUT
    spec = W.MultiSpec("spec_n20_t2_h24_wait", N=20, T=2, H=24, num_slots=70, seed=330)
    x = W.make_multi_inputs(spec)
    d = _dev(x, cuda_device)
    wq = torch.zeros(2, dtype=torch.int32, device=cuda_device)
    _call(x, d, queue=wq).wait_test(20_000_000, withhold_unit=x.N * x.H - 3)
    torch.cuda.synchronize()
    assert int(d["err_flag"].item()) & KDA_DEVERR_TIMEOUT
    assert wq.tolist() == [0, 0]
    y = W.make_multi_inputs(W.MultiSpec("spec_n5_t2_h12_after", N=5, T=2, H=12, num_slots=20, seed=331))
    dy = _dev(y, cuda_device)
    _call(y, dy)()
    _compare(y, dy, _oracle(y))


def test_bench_batch_sampled(cuda_device):
    """The measured batch (64 sequences of 4 tokens, H = 48, 4 padding
    sequences) in the launch configuration the benchmark times (work queue,
    graph replay), against the oracle."""
    from linear_attention_decode_04_gb300.stack import warm_up
    x = W.make_multi_inputs(W.MULTI_BENCH)
    d = _dev(x, cuda_device)
    wq = torch.zeros(2, dtype=torch.int32, device=cuda_device)
    c = _call(x, d, queue=wq)
    warm_up(cuda_device)
    s = torch.cuda.Stream(cuda_device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c()
    g.replay()
    _compare(x, d, _oracle(x))
