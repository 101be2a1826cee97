"""A decode step over a stack of independent KDA layers, replayed as one CUDA
graph.

P1 ("[ROCm][Perf] Kimi-K3 Fused kernel for KDA decode", 执行摘要 and
实现拆解 item 5) argues that eager timing overstates the gain of fusing the
decode chain and that CUDA-graph replay of one step across the model's 69
KDA layers is the measurement that decides.  ``DecodeStack`` captures one
``kda_decode`` launch per layer, each with its own weights, conv state and
recurrent-state pool, into a single graph; replaying it advances every
layer's state by one token.
"""
from __future__ import annotations

import torch

from .binding import KdaDecodeCall, kda_decode

# per-token inputs of a layer (copied in each step); the rest is resident
STEP_INPUTS = ("qkv", "g", "beta", "gate", "slot_idx")


def warm_up(device: torch.device) -> None:
    """Launch every kernel variant once on a one-row padding problem (writes
    only a zero output row), so that kernel loading and the library's
    once-per-device set-up happen before any stream capture."""
    dev = torch.device(device)
    z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=dev)  # noqa: E731
    for out_norm in (True, False):
        for upd in (True, False):
            kda_decode(z(1, 384, dt=torch.bfloat16), z(3, 4, 128), z(1, 384, 3, dt=torch.bfloat16),
                       z(1, 1, 128, 128), z(1, 1, 128), z(1, 1, dt=torch.bfloat16),
                       z(1, dt=torch.int32), z(1, 128, dt=torch.bfloat16),
                       gate=z(1, 128, dt=torch.bfloat16), norm_weight=z(128),
                       out_norm=out_norm, update_conv_state=upd)
    torch.cuda.synchronize(dev)


class DecodeStack:
    """``layers`` is a list of dicts of device tensors with the keys of
    ``kda_decode`` (qkv, conv_weight, conv_state, state, g, beta, slot_idx,
    out, gate, norm_weight, conv_bias, err_flag).  With ``host_token_io`` the
    per-token tensors (``STEP_INPUTS`` and out) may be pinned host tensors,
    read and written by the kernels directly over the CPU-GPU link, so a step
    needs no copies at all.  Each layer must own its
    state and conv-state pools.  With two or more layers, consecutive launches
    never share a pool (the last layer is followed by the first on the next
    replay), so every launch may stream its state while the previous layer's
    kernel drains (KDA_EARLY_PREFETCH)."""

    def __init__(self, layers: list[dict], eps: float = 1e-6, out_norm: bool = True,
                 update_conv_state: bool = True, host_token_io: bool = False,
                 work_queue: bool | None = None):
        self.layers = layers
        ptrs = [L["state"].data_ptr() for L in layers]
        if len(set(ptrs)) != len(ptrs):
            raise ValueError("every layer needs its own state pool")
        early = len(layers) > 1
        # Every launch takes the dynamic schedule (work queue): each CTA takes a
        # static prefix of its units and draws the rest from the queue, so the
        # CTAs end together (measured on GB300: 64.26 -> 63.95 us per launch of
        # a 20-layer stack against the purely static schedule, 516 -> 507 us on
        # an N = 256, H = 96 launch).  One queue serves every layer: the
        # launches are ordered on one stream and each touches the queue only
        # after the previous one ended.  ``work_queue=False`` keeps the static
        # schedule.
        dev = layers[0]["state"].device
        use_queue = True if work_queue is None else bool(work_queue)
        self.queue = torch.zeros(2, dtype=torch.int32, device=dev) if use_queue else None
        self.calls = [
            KdaDecodeCall(L["qkv"], L["conv_weight"], L["conv_state"], L["state"], L["g"], L["beta"],
                          L["slot_idx"], L["out"], gate=L.get("gate"),
                          norm_weight=L.get("norm_weight"), conv_bias=L.get("conv_bias"), eps=eps,
                          out_norm=out_norm, update_conv_state=update_conv_state,
                          err_flag=L.get("err_flag"), early_prefetch=early,
                          work_queue=self.queue, host_token_io=host_token_io)
            for L in layers
        ]
        self.graph: torch.cuda.CUDAGraph | None = None
        self.stream: torch.cuda.Stream | None = None

    @property
    def launches_per_step(self) -> int:
        return len(self.calls)

    def run_eager(self, stream: torch.cuda.Stream | None = None) -> None:
        for c in self.calls:
            c(stream)

    def capture(self, stream: torch.cuda.Stream | None = None) -> torch.cuda.CUDAGraph:
        dev = self.layers[0]["state"].device
        warm_up(dev)
        self.stream = stream if stream is not None else torch.cuda.Stream(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for c in self.calls:
                c()
        self.graph = g
        return g

    def replay(self) -> None:
        self.graph.replay()
