"""One MXFP8 MoE FFN layer training step (forward + backward) over preallocated device buffers.

This composes the C-ABI calls of the hot path in the order the pages describe
(aigc.bar "Blackwell性能陷阱？…MoE提速3.5倍的底层逻辑", section "2. 被忽视的“量化税”":
quantize the inputs, then the grouped matmuls; backward needs a transpose-quantize
as well):

forward   weights W1 [E, 2I, H], W2 [E, H, I] quantized rowwise and columnwise in one
          read each; routing ids permuted by expert; activations x [T, H] quantized on
          gather (read once in expert order -> rowwise GEMM1 operand and columnwise
          wgrad1 operand); GEMM1 (x W1_e^T -> [gate | up] [R, 2I]); SwiGLU fused with
          quantization: h = silu(gate) * up straight to the rowwise GEMM2 operand and the
          columnwise wgrad2 operand; GEMM2 (h W2_e^T -> Y [R, H]); combine:
          out[t] = sum_j gate_w[t][j] Y[dst_of[t][j]] (bf16 [T, H], back in token order).
backward  combine backward: dgate [T, k] and each routed row's gate; dY [R, H] = bf16(gate * dOut)
          formed on the fly by quantize-on-gather of dOut with the gate as a row scale, rowwise +
          columnwise, never written in bf16 (fuse_dy=False: combine backward writes the routed
          bf16 dY, then a plain quantize -- same bytes); dgrad2 (dY W2_e -> [R, I]); wgrad2 (dY_e^T h_e -> fp32
          [E, H, I]); SwiGLU backward fused with quantization: dH [R, 2I] from dh and the
          saved GEMM1 output straight to the rowwise dgrad1 operand and the columnwise wgrad1
          operand; dgrad1 (dH W1_e -> [R, H]);
          wgrad1 (dH_e^T x_e -> fp32 [E, 2I, H]); un-permute sum of the input gradient
          dx[t] = sum_j dX[dst_of[t][j]] (bf16 [T, H]).

The layer's own inputs (x, ids, gate, dOut) and outputs (out, dx) are in token order;
the weight gradients dW1, dW2 and dgate stay on the device.  Everything runs on the
current torch stream; nothing synchronizes.
"""
from __future__ import annotations

import torch

from . import binding as mx


class MoEFFNStep:
    """Buffers and launch sequence of one MoE FFN forward+backward step."""

    def __init__(self, T: int, E: int, k: int, hidden: int, inter: int, device="cuda", fuse_swiglu: bool = False,
                 fuse_dy: bool = True):
        """fuse_swiglu: GEMM1 and SwiGLU + quantization in one launch (grouped_gemm_mxfp8_fwd_swiglu)
        instead of grouped_gemm_mxfp8_fwd followed by mxfp8_swiglu_quantize; same outputs.
        fuse_dy: the output gradient dY quantized on the fly from dOut (no bf16 dY, the default);
        False: combine backward writes the routed bf16 dY and a plain quantize reads it back; same
        outputs.  At the MoE FFN shape the fused form takes 0.37 + 0.64 ms against 0.67 + 0.59 ms
        (its quantize-on-gather reads dOut from L2 for most slots)."""
        self.T, self.E, self.k, self.H, self.I = T, E, k, hidden, inter
        self.fuse_swiglu = fuse_swiglu
        self.fuse_dy = fuse_dy
        self.I2 = 2 * inter
        self.R = R = T * k
        dev = torch.device(device)
        self.dev = dev
        H, I, I2 = hidden, inter, 2 * inter
        u8, bf, i32, f32 = torch.uint8, torch.bfloat16, torch.int32, torch.float32
        pb = mx.mx_padded_rows_bound(R, E)
        self.pb = pb
        sfb = mx.mx_sf_bytes
        sfb4 = mx.mx_sf_bytes_x4   # B operands of the grouped GEMMs take their scales in the four-copy layout

        def z(*shape, dtype=u8):
            return torch.empty(*shape, dtype=dtype, device=dev)

        # inputs (filled by the caller)
        self.x = z(T, H, dtype=bf)
        self.ids = z(T, k, dtype=i32)
        self.gate = z(T, k, dtype=f32)
        self.dout = z(T, H, dtype=bf)
        self.w1 = z(E, I2, H, dtype=bf)
        self.w2 = z(E, H, I, dtype=bf)
        # weights: rowwise (forward B) and columnwise (dgrad B), experts as 128-aligned segments
        self.w1_q, self.w1_sf = z(E * I2, H), z(sfb4(E * I2, H // 32))
        self.w1c_q, self.w1c_sf = z(H, E * I2), z(sfb4(H, E * I2 // 32))
        self.w2_q, self.w2_sf = z(E * H, I), z(sfb4(E * H, I // 32))
        self.w2c_q, self.w2c_sf = z(I, E * H), z(sfb4(I, E * H // 32))
        self.w1_seg = torch.arange(0, (E + 1) * I2, I2, dtype=i32, device=dev)
        self.w2_seg = torch.arange(0, (E + 1) * H, H, dtype=i32, device=dev)
        # activations
        self.counts, self.off, self.poff = z(E, dtype=i32), z(E + 1, dtype=i32), z(E + 1, dtype=i32)
        self.src_row, self.dst_of = z(R, dtype=i32), z(R, dtype=i32)
        self.ws_bytes = mx.moe_permute_workspace_bytes(T, k, E)
        self.ws = z(max(self.ws_bytes, 16))
        self.a1_q, self.a1_sf = z(R, H), z(sfb(pb, H // 32))
        self.out1 = z(R, I2, dtype=bf)
        self.h_q, self.h_sf = z(R, I), z(sfb(pb, I // 32))
        self.hc_q, self.hc_sf = z(I, pb), z(sfb4(I, pb // 32))   # wgrad2 B
        self.out2 = z(R, H, dtype=bf)
        self.out = z(T, H, dtype=bf)
        # backward
        self.dy = z(R, H, dtype=bf) if not fuse_dy else None   # materialized only without fuse_dy
        self.dgate = z(T, k, dtype=f32)
        self.gate_rows = z(R, dtype=f32)                         # routing weight of each routed row
        self.dy_q, self.dy_sf = z(R, H), z(sfb(pb, H // 32))
        self.dyc_q, self.dyc_sf = z(H, pb), z(sfb(H, pb // 32))
        self.dh_q, self.dh_sf = z(R, I2), z(sfb(pb, I2 // 32))
        self.dhc_q, self.dhc_sf = z(I2, pb), z(sfb(I2, pb // 32))
        self.xpc_q, self.xpc_sf = z(H, pb), z(sfb4(H, pb // 32))   # wgrad1 B
        self.dh_in = z(R, I, dtype=bf)
        self.dx_routed = z(R, H, dtype=bf)
        self.dx = z(T, H, dtype=bf)
        self.dw2 = z(E, H, I, dtype=f32)
        self.dw1 = z(E, I2, H, dtype=f32)
        self.dev_err = torch.zeros(1, dtype=i32, device=dev)
        self.gemm_hook = None      # optional callable(name, flops, fn) wrapping each GEMM launch
        self.launches = 0          # CUDA kernels launched by this object

    # ------------------------------------------------------------------ helpers
    def gemm_flops(self):
        R, H, I, I2 = self.R, self.H, self.I, self.I2
        return {"fwd1": 2 * R * I2 * H, "fwd2": 2 * R * H * I, "dgrad2": 2 * R * I * H,
                "wgrad2": 2 * R * H * I, "dgrad1": 2 * R * H * I2, "wgrad1": 2 * R * I2 * H}

    def _gemm(self, name, fn):
        self.launches += 1
        if self.gemm_hook is None:
            fn()
        else:
            self.gemm_hook(name, self.gemm_flops()[name], fn)

    def _quant(self, x, rows, cols, mode, seg, nseg, ld, q_row, sf_row, q_col, sf_col):
        self.launches += 1
        mx.mxfp8_quantize(x, rows, cols, mode, seg[0] if seg else None, seg[1] if seg else None, nseg, ld,
                          q_row, sf_row, q_col, sf_col, self.dev_err)

    # ------------------------------------------------------------------ the step
    def forward(self, before_inputs=None):
        """The forward launches.  before_inputs: called (on the host, in launch order) after the
        weight quantization and before the first launch that reads ids, gate or x -- e.g. a stream
        wait on the event that marks their arrival, so that the weights are quantized while the
        inputs are still being copied."""
        T, E, k, H, I, I2, R, pb = self.T, self.E, self.k, self.H, self.I, self.I2, self.R, self.pb
        RC = mx.MX_ROWWISE | mx.MX_COLWISE
        RC_B = RC | mx.MX_ROWWISE_X4 | mx.MX_COLWISE_X4   # both forms are B operands
        RC_CB = RC | mx.MX_COLWISE_X4                     # rowwise A operand, columnwise B operand
        self._quant(self.w1, E * I2, H, RC_B, (self.w1_seg, self.w1_seg), E, E * I2,
                    self.w1_q, self.w1_sf, self.w1c_q, self.w1c_sf)
        self._quant(self.w2, E * H, I, RC_B, (self.w2_seg, self.w2_seg), E, E * H,
                    self.w2_q, self.w2_sf, self.w2c_q, self.w2c_sf)
        if before_inputs is not None:
            before_inputs()
        self.launches += 3
        mx.moe_permute(self.ids, T, k, E, self.counts, self.off, self.poff, self.src_row, self.dst_of,
                       None, None, 0, None, None, self.ws, self.ws_bytes, self.dev_err)
        # quantize-on-gather: x read once in expert order -> rowwise GEMM1 operand and the
        # columnwise wgrad1 operand
        self.launches += 1
        mx.mxfp8_gather_quantize(self.x, T, H, RC_CB, self.src_row, self.off, self.poff, E, R, pb,
                                 self.a1_q, self.a1_sf, self.xpc_q, self.xpc_sf, self.dev_err)
        if self.fuse_swiglu:
            self._gemm("fwd1", lambda: mx.grouped_gemm_mxfp8_fwd_swiglu(
                self.a1_q, self.a1_sf, self.w1_q, self.w1_sf, self.off, self.poff, E, R, I, H, self.out1, self.h_q,
                self.h_sf, self.hc_q, self.hc_sf, pb, RC_CB, self.dev_err))
        else:
            self._gemm("fwd1", lambda: mx.grouped_gemm_mxfp8_fwd(self.a1_q, self.a1_sf, self.w1_q, self.w1_sf,
                                                                 self.off, self.poff, E, R, I2, H, self.out1,
                                                                 self.dev_err))
            self.launches += 1
            mx.mxfp8_swiglu_quantize(self.out1, R, I, RC_CB, self.off, self.poff, E, pb, self.h_q, self.h_sf, self.hc_q,
                                     self.hc_sf, self.dev_err)
        self._gemm("fwd2", lambda: mx.grouped_gemm_mxfp8_fwd(self.h_q, self.h_sf, self.w2_q, self.w2_sf, self.off,
                                                             self.poff, E, R, H, I, self.out2, self.dev_err))
        self.launches += 1
        mx.moe_combine_fwd(self.out2, self.gate, self.dst_of, T, k, H, R, self.out, self.dev_err)

    def backward(self):
        T, k, E, H, I, I2, R, pb = self.T, self.k, self.E, self.H, self.I, self.I2, self.R, self.pb
        RC = mx.MX_ROWWISE | mx.MX_COLWISE
        if self.fuse_dy:
            self.launches += 2
            mx.moe_combine_bwd_ex(self.dout, self.out2, self.gate, self.dst_of, T, k, H, R, None, self.dgate,
                                  self.gate_rows, self.dev_err)
            mx.mxfp8_gather_quantize_ex(self.dout, T, H, RC, self.src_row, self.gate_rows, self.off, self.poff, E, R,
                                        pb, self.dy_q, self.dy_sf, self.dyc_q, self.dyc_sf, self.dev_err)
        else:
            self.launches += 1
            mx.moe_combine_bwd(self.dout, self.out2, self.gate, self.dst_of, T, k, H, R, self.dy, self.dgate,
                               self.dev_err)
            self._quant(self.dy, R, H, RC, (self.off, self.poff), E, pb, self.dy_q, self.dy_sf, self.dyc_q,
                        self.dyc_sf)
        self._gemm("dgrad2", lambda: mx.grouped_gemm_mxfp8_dgrad(self.dy_q, self.dy_sf, self.w2c_q, self.w2c_sf,
                                                                 self.off, self.poff, E, R, I, H, self.dh_in,
                                                                 self.dev_err))
        self._gemm("wgrad2", lambda: mx.grouped_gemm_mxfp8_wgrad(self.dyc_q, self.dyc_sf, self.hc_q, self.hc_sf,
                                                                 self.off, self.poff, E, H, I, pb, self.dw2,
                                                                 self.dev_err))
        self.launches += 1
        mx.mxfp8_swiglu_bwd_quantize(self.dh_in, self.out1, R, I, RC, self.off, self.poff, E, pb, self.dh_q,
                                     self.dh_sf, self.dhc_q, self.dhc_sf, self.dev_err)
        self._gemm("dgrad1", lambda: mx.grouped_gemm_mxfp8_dgrad(self.dh_q, self.dh_sf, self.w1c_q, self.w1c_sf,
                                                                 self.off, self.poff, E, R, H, I2, self.dx_routed,
                                                                 self.dev_err))
        self._gemm("wgrad1", lambda: mx.grouped_gemm_mxfp8_wgrad(self.dhc_q, self.dhc_sf, self.xpc_q, self.xpc_sf,
                                                                 self.off, self.poff, E, I2, H, pb, self.dw1,
                                                                 self.dev_err))
        self.launches += 1
        mx.moe_combine_fwd(self.dx_routed, None, self.dst_of, T, k, H, R, self.dx, self.dev_err)

    def step(self):
        self.forward()
        self.backward()

    def capture(self, stream=None):
        """Record one whole step (forward + backward, every launch on the buffers above) as a
        CUDA graph and return it; `graph.replay()` then reruns the step without per-launch host
        work.  One eager step must have run on this device first (the grouped GEMM sets its
        shared-memory attribute on its first launch there, which a capture cannot hold).
        Inputs are read from, and outputs written to, the same buffers as `step()`, so new inputs
        go in with `copy_` into `x`, `ids`, `gate`, `dout`, `w1`, `w2` before a replay."""
        s = torch.cuda.Stream(device=self.dev) if stream is None else stream
        s.wait_stream(torch.cuda.current_stream(self.dev))
        graph = torch.cuda.CUDAGraph()
        hook, self.gemm_hook = self.gemm_hook, None
        try:
            with torch.cuda.graph(graph, stream=s):
                self.step()
        finally:
            self.gemm_hook = hook
        torch.cuda.current_stream(self.dev).wait_stream(s)
        return graph
