"""One transformer block's linear sites on one denoising step, in the
precision the step policy picks: the call sequence of the step-scheduled
stack, over the C ABI.

This module only orders calls, owns the buffers they write and the streams
they overlap on; every value is computed by the library's kernels.

A W8A8 step (the middle steps, diffusers PR #14664, "[Cosmos3] Mixed
W8A8/W8A16 denoising for ModelOpt FP8 checkpoints", section Behavior):
  qkv_shared_quant_gemm   Q/K/V, one shared quantization of the block input
  fp8_quant_static        the out-projection's and the MLP's inputs, on a
                          side stream while the Q/K/V GEMM runs (they do not
                          depend on it)
  fp8_linear_w8a8         out-projection on those codes
  gate_up_swiglu_fp8      gate/up with SiLU(gate) * up written to E4M3 in the
                          GEMM epilogue (TensorRT-LLM PR #17476, "Load static
                          FP8 Cosmos3 Nano/Super checkpoints without
                          re-quantizing them", section What changed)
  fp8_linear_w8a8         down projection on the E4M3 codes
A W8A16 step (the first and last steps: "dequant + F.linear"): the block's
seven weights are dequantized on a side stream in the order the GEMMs need
them (weights do not depend on activations), and each site runs the bf16
GEMM on its dequantized weight as soon as that is ready; gate/up run with
the bf16 SwiGLU fused into their epilogue.
"""

from dataclasses import dataclass
from typing import List, Tuple

import torch


@dataclass
class BlockWeights:
    """E4M3 weights ``[N, K]`` (uint8) with their one-element float32 scales,
    and the static input scales of the block's sites."""
    qkv: List[Tuple[torch.Tensor, torch.Tensor]]      # 3 x ([H, H], s_w)
    out: Tuple[torch.Tensor, torch.Tensor]            # [H, H]
    gu: List[Tuple[torch.Tensor, torch.Tensor]]       # gate, up: [I, H]
    down: Tuple[torch.Tensor, torch.Tensor]           # [H, I]
    s_qkv: torch.Tensor                               # input scale of Q/K/V
    s_out: torch.Tensor                               # input scale of the out-projection
    s_mlp: torch.Tensor                               # input scale of gate/up
    s_h: torch.Tensor                                 # input scale of down (SwiGLU output)


class BlockStep:
    """Buffers and streams for running blocks of ``M`` tokens, hidden ``H``
    and intermediate ``I`` on one device.  Outputs of the last run stay in
    ``y_qkv``, ``y_out``, ``h8`` (W8A8) or ``h16`` (W8A16), ``y_down``."""

    def __init__(self, M, H, I, device):
        self.M, self.H, self.I, self.dev = M, H, I, device
        bf = dict(dtype=torch.bfloat16, device=device)
        u8 = dict(dtype=torch.uint8, device=device)
        self.y_qkv = [torch.empty((M, H), **bf) for _ in range(3)]
        self.y_out = torch.empty((M, H), **bf)
        self.y_down = torch.empty((M, H), **bf)
        self.h8 = torch.empty((M, I), **u8)
        self.h16 = torch.empty((M, I), **bf)
        self.ws = torch.empty((M, H), **u8)
        self.q_out = torch.empty((M, H), **u8)
        self.q_mlp = torch.empty((M, H), **u8)
        self._y_gu = None
        # transient bf16 weights of every site of a block (W8A16 steps)
        shapes = [(H, H)] * 4 + [(I, H)] * 2 + [(H, I)]
        wd_all = torch.empty((sum(n * k for n, k in shapes),), **bf)
        views, off = [], 0
        for n, k in shapes:
            views.append(wd_all[off:off + n * k].view(n, k))
            off += n * k
        self.wd_qkv, self.wd_out, self.wd_gu, self.wd_down = views[:3], views[3], views[4:6], views[6]
        self.side = torch.cuda.Stream(device=device)
        self.dq = torch.cuda.Stream(device=device)
        self.dq_ev = [torch.cuda.Event() for _ in range(4)]

    @property
    def y_gu(self):
        """bf16 gate/up outputs of the unfused MLP form (allocated on first use)."""
        if self._y_gu is None:
            self._y_gu = [torch.empty((self.M, self.I), dtype=torch.bfloat16, device=self.dev)
                          for _ in range(2)]
        return self._y_gu

    def outputs(self):
        return self.y_qkv + [self.y_out, self.y_down]

    def run(self, W, mode, w, x_qkv, x_out, x_mlp, fused=True):
        """One block pass in ``mode`` (W.MODE_A8 / W.MODE_A16) on the current
        stream; returns the number of kernel launches it enqueues.  ``fused``
        selects the fused gate/up + SwiGLU kernel, else the group GEMM
        followed by the SwiGLU kernel."""
        wq, sq = [q for q, _ in w.qkv], [s for _, s in w.qkv]
        wgu, sgu = [q for q, _ in w.gu], [s for _, s in w.gu]
        main = torch.cuda.current_stream()
        if mode == W.MODE_A8:
            self.side.wait_stream(main)
            with torch.cuda.stream(self.side):
                W.fp8_quant_static(x_out, w.s_out, out=self.q_out)
                W.fp8_quant_static(x_mlp, w.s_mlp, out=self.q_mlp)
            W.qkv_shared_quant_gemm(W.MODE_A8, x_qkv, w.s_qkv, wq, sq, outs=self.y_qkv, ws=self.ws)
            main.wait_stream(self.side)
            W.fp8_linear_w8a8(self.q_out, w.out[0], w.s_out, w.out[1], out=self.y_out)
            if fused:
                W.gate_up_swiglu_fp8(self.q_mlp, w.s_mlp, wgu[0], wgu[1], sgu[0], sgu[1], w.s_h, out=self.h8)
            else:
                W.fp8_linear_w8a8_group(self.q_mlp, w.s_mlp, wgu, sgu, outs=self.y_gu)
                W.swiglu_2in_fp8(self.y_gu[0], self.y_gu[1], w.s_h, out=self.h8)
            W.fp8_linear_w8a8(self.h8, w.down[0], w.s_h, w.down[1], out=self.y_down)
            return 7 if fused else 8
        # dequant + F.linear, scheduled: the previous step's GEMMs must be done
        # with the dequantized-weight buffers before they are overwritten
        self.dq.wait_stream(main)
        sites = [(list(zip(wq, sq)), self.wd_qkv), ([w.out], [self.wd_out]),
                 (list(zip(wgu, sgu)), self.wd_gu), ([w.down], [self.wd_down])]
        with torch.cuda.stream(self.dq):
            for (ws_, outs_), ev in zip(sites, self.dq_ev):
                for (q, sc), o in zip(ws_, outs_):
                    W.fp8_dequant_weight(q, sc, out=o)
                ev.record(self.dq)
        main.wait_event(self.dq_ev[0])
        W.bf16_linear_group(x_qkv, self.wd_qkv, outs=self.y_qkv)
        main.wait_event(self.dq_ev[1])
        W.bf16_linear_group(x_out, [self.wd_out], outs=[self.y_out])
        main.wait_event(self.dq_ev[2])
        if fused:
            W.bf16_gate_up_swiglu(x_mlp, self.wd_gu[0], self.wd_gu[1], out=self.h16)
        else:
            W.bf16_linear_group(x_mlp, self.wd_gu, outs=self.y_gu)
            W.swiglu_2in_bf16(self.y_gu[0], self.y_gu[1], out=self.h16)
        main.wait_event(self.dq_ev[3])
        W.bf16_linear_group(self.h16, [self.wd_down], outs=[self.y_down])
        return 11 if fused else 12
