"""One routed-expert MLP layer on one GPU: device buffers plus the sequence
of C-ABI calls that makes a forward and a backward pass.

Torch is used only to allocate device memory and to name the stream; every
step of the path runs in libmoe's kernels.  All buffers are allocated once
for the worst case (capacity = T*k + E*127 rows), so a whole step can be
captured in one CUDA graph and replayed with no host synchronisation.
"""
from __future__ import annotations

import contextlib
import math

import torch

from . import _lib as L


class MoEExpertMLP:
    def __init__(self, E, d, F, T=0, k=1, act="swiglu", alpha=1.0, limit=math.inf,
                 linear_offset=0.0, out_scale=1.0, has_b1=False, has_b2=False, sm_margin=0,
                 capacity=None, device="cuda", recompute_h=False, dtype="bf16",
                 keep_bf16_copies=None):
        self.desc = L.make_desc(T, E, k, d, F, act=act, alpha=alpha, limit=limit,
                                linear_offset=linear_offset, out_scale=out_scale,
                                has_b1=has_b1, has_b2=has_b2, sm_margin=sm_margin,
                                capacity=capacity, recompute_h=recompute_h, dtype=dtype)
        # dtype "mxfp8": the grouped GEMMs read MXFP8 operands (E4M3 codes,
        # E8M0 scales per 32 elements); routing and combine stay bf16
        self.mx = dtype == "mxfp8"
        # dtype "nvfp4": packed E2M1 operands with UE4M3 scales per 16
        # elements and per-tensor encode scales from their amax
        self.nv = dtype == "nvfp4"
        # dtype "fp32": fp32 tensors throughout, GEMMs on the TF32 tensor
        # cores; the backward reads transposed copies (weights transposed
        # once per load, A and dH^T by their epilogues, x_perm and dY by a
        # transpose pass)
        self.f32 = dtype == "fp32"
        if self.f32 and recompute_h:
            raise ValueError("recompute_h is not supported with fp32 tensors")
        # optional fused NVFP4-preparation outputs (per-tensor amax of A and
        # of dH, plain and Hadamard-rotated): float[2] device tensors or None
        self.amax_a = None
        self.amax_dh = None
        # recompute_h: the forward keeps no H; the backward regenerates it in
        # the library workspace (activation recompute)
        self.recompute_h = recompute_h
        # the bf16 A and dH: on the MXFP8 path the later GEMMs read only
        # their MXFP8 copies, so by default they are not written there (dH
        # still is when the FC1 bias gradient needs it); the bf16 and NVFP4
        # paths always write them
        self.keep_bf16 = (dtype != "mxfp8") if keep_bf16_copies is None else bool(keep_bf16_copies)
        # MXFP8: whether the rowwise copies of x_perm / dY were written by the
        # permutation / the combine backward (then the quantize passes make
        # only the transposed copies)
        self._x_row_fused = False
        self._dy_row_fused = False
        self.T, self.E, self.k, self.d, self.F = T, E, k, d, F
        self.Fp = L.moe_fc1_padded_width(F)
        # FC1 output width: packed gate|linear halves (2*F_pad) for the GLU
        # activations, F for the non-gated squared ReLU
        self.W1 = F if act == "srelu" else 2 * self.Fp
        self.gated = act != "srelu"
        self.has_b1, self.has_b2 = has_b1, has_b2
        cap = self.desc.capacity
        self.capacity = cap
        dev = torch.device(device)
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        if self.f32:
            bf = f32          # every activation, weight and gradient tensor
        self.act_dtype = bf

        def z(*shape, dtype=bf):
            return torch.zeros(shape, dtype=dtype, device=dev)

        # weights (FC1 kept repacked) and their gradients
        self.w1p = z(E, self.W1, d)
        self.b1p = z(E, self.W1) if has_b1 else None
        self.w2 = z(E, d, F)
        self.b2 = z(E, d) if has_b2 else None
        self.dw1p = z(E, self.W1, d)
        self.db1p = z(E, self.W1) if has_b1 else None
        self.dw2 = z(E, d, F)
        self.db2 = z(E, d) if has_b2 else None
        # routing state (device resident)
        self.topk_idx = z(max(T, 1), k, dtype=i32)
        self.topk_w = z(max(T, 1), k, dtype=f32)
        self.counts = z(E, dtype=i32)
        self.offsets = z(E + 1, dtype=i32)
        self.padded_offsets = z(E + 1, dtype=i32)
        self.tile_prefix = z(E + 1, dtype=i32)
        self.row_src = z(cap, dtype=i32)
        self.row_of = z(max(T, 1), k, dtype=i32)
        # per-row activations and gradients (padded row layout)
        self.x_perm = z(cap, d)
        self.h = None if recompute_h else z(cap, self.W1)
        self.a = z(cap, F)
        self.y = z(cap, d)
        self.dy = z(cap, d)
        self.dh = z(cap, self.W1)
        self.dx_perm = z(cap, d)
        # per-token outputs
        self.out = z(max(T, 1), d)
        self.dw = z(max(T, 1), k, dtype=f32)
        self.dx = z(max(T, 1), d)
        self.dlogits = z(max(T, 1), E, dtype=f32)
        self.ws = torch.zeros(max(L.moe_workspace_size(self.desc), 256), dtype=torch.uint8, device=dev)
        if self.f32:
            self.w1t = z(E, d, self.W1)
            self.w2t = z(E, F, d)
            self.x_t = z(d, cap)
            self.a_t = z(F, cap)
            self.dy_t = z(d, cap)
            self.dh_t = z(self.W1, cap)
        if self.mx:
            # activations: rowwise for the GEMM that contracts over features,
            # transposed for the weight gradient that contracts over rows
            self.x_mx = self.mx_operand(d)
            self.a_mx = self.mx_operand(F)
            self.dy_mx = self.mx_operand(d)
            self.dh_mx = self.mx_operand(self.W1)
            u8 = torch.uint8

            def sc(rows, cols):
                return z(E * L.moe_mx_scale_bytes(rows, cols), dtype=u8)

            W1 = self.W1
            self.w_mx = dict(w1=z(E, W1, d, dtype=u8), w1_s=sc(W1, d),
                             w1t=z(E, d, W1, dtype=u8), w1t_s=sc(d, W1),
                             w2=z(E, d, F, dtype=u8), w2_s=sc(d, F),
                             w2t=z(E, F, d, dtype=u8), w2t_s=sc(F, d))

        if self.nv:
            # activations: rowwise for the GEMM that contracts over features,
            # the rotated transposed copy for the weight gradient
            self.x_nv = self.nv_operand(d)
            self.a_nv = self.nv_operand(F)
            self.dy_nv = self.nv_operand(d)
            self.dh_nv = self.nv_operand(self.W1)
            u8 = torch.uint8

            def scn(rows, cols):
                return z(E * L.moe_nvfp4_scale_bytes(rows, cols), dtype=u8)

            W1 = self.W1
            self.w_nv = dict(w1=z(E, W1, d // 2, dtype=u8), w1_s=scn(W1, d),
                             w1t=z(E, d, W1 // 2, dtype=u8), w1t_s=scn(d, W1),
                             w2=z(E, d, F // 2, dtype=u8), w2_s=scn(d, F),
                             w2t=z(E, F, d // 2, dtype=u8), w2t_s=scn(F, d),
                             amax=z(4, dtype=f32))

    def nv_operand(self, width):
        """NVFP4 buffers of a per-row tensor [capacity, width]: packed rowwise
        codes + scales, the rotated transposed copy, and its encode amax pair
        (plain, rotated)."""
        cap, dev, u8 = self.capacity, self.w2.device, torch.uint8
        return dict(q=torch.zeros((cap, width // 2), dtype=u8, device=dev),
                    scale=torch.zeros(L.moe_nvfp4_scale_bytes(cap, width), dtype=u8, device=dev),
                    qt=torch.zeros((width, cap // 2), dtype=u8, device=dev),
                    scale_t=torch.zeros(L.moe_nvfp4_scale_bytes(width, cap), dtype=u8,
                                        device=dev),
                    amax=torch.zeros(2, dtype=torch.float32, device=dev), layout="mma")

    def mx_operand(self, width):
        """MXFP8 buffers of a per-row tensor [capacity, width] in the MMA scale
        layout: rowwise codes + scales and the transposed copy.  Scale
        buffers start zeroed (entries past the tensor are read, never
        written)."""
        cap, dev, u8 = self.capacity, self.w2.device, torch.uint8
        return dict(q=torch.zeros((cap, width), dtype=u8, device=dev),
                    scale=torch.zeros(L.moe_mx_scale_bytes(cap, width), dtype=u8, device=dev),
                    qt=torch.zeros((width, cap), dtype=u8, device=dev),
                    scale_t=torch.zeros(L.moe_mx_scale_bytes(width, cap), dtype=u8, device=dev),
                    layout="mma")

    # ------------------------------------------------------------ weights
    def load_weights(self, w1, b1, w2, b2, stream=None):
        """w1 [E,2F,d] logical (gate rows then linear rows), b1 [E,2F], w2
        [E,d,F], b2 [E,d]; bf16 device tensors.  FC1 is repacked on device."""
        L.moe_repack_fc1(self.desc, w1, b1 if self.has_b1 else None, self.w1p,
                         self.b1p if self.has_b1 else None, stream)
        self.w2.copy_(w2)
        if self.has_b2:
            self.b2.copy_(b2)
        if self.mx or self.nv:
            self.quantize_weights(stream)
        if self.f32:
            L.moe_transpose_weights_tf32(self.desc, self.w1p, self.w2, self.w1t, self.w2t, stream)

    def quantize_weights(self, stream=None):
        """MXFP8 / NVFP4 weight copies (rowwise and transposed) from the bf16
        masters; once per optimizer step."""
        if self.nv:
            L.moe_quantize_weights_nvfp4(self.desc, self.w1p, self.w2, self.w_nv, stream)
        else:
            L.moe_quantize_weights_mx(self.desc, self.w1p, self.w2, self.w_mx, stream)

    def unpack_fc1(self, packed, width, stream=None):
        """Packed [E,2F_pad,width] -> logical [E,2F,width] (e.g. dW1p, db1p);
        [E,F,width] unchanged for the non-gated activation."""
        n1 = 2 * self.F if self.gated else self.F
        out = torch.empty((self.E, n1, width), dtype=self.act_dtype, device=packed.device)
        L.moe_unpack_fc1(self.desc, packed, out, width, stream)
        return out

    # ------------------------------------------------------------ passes
    # Each pass below is a fixed sequence of C-ABI calls.  `timer`, if given,
    # is a callable name -> context manager wrapped around each call (used by
    # the benchmark to time individual kernels); it does no work itself.
    @staticmethod
    def _t(timer, name):
        return timer(name) if timer is not None else contextlib.nullcontext()

    def route(self, x, logits, bias=None, stream=None, timer=None):
        with self._t(timer, "route_permute"):
            if self.mx:          # x_perm's rowwise MXFP8 copy written by the gather
                L.moe_route_permute_mx(self.desc, logits, bias, x, self.topk_idx, self.topk_w,
                                       self.counts, self.offsets, self.padded_offsets,
                                       self.tile_prefix, self.row_src, self.row_of, self.x_perm,
                                       self._rowwise(self.x_mx), self.ws, stream)
                self._x_row_fused = True
            else:
                L.moe_route_permute(self.desc, logits, bias, x, self.topk_idx, self.topk_w,
                                    self.counts, self.offsets, self.padded_offsets,
                                    self.tile_prefix, self.row_src, self.row_of, self.x_perm,
                                    self.ws, stream)

    @staticmethod
    def _rowwise(mx):
        return dict(q=mx["q"], scale=mx["scale"], layout="mma")

    @staticmethod
    def _colwise(mx):
        return dict(qt=mx["qt"], scale_t=mx["scale_t"], layout="mma")

    def route_fused(self, x, w_router, bias=None, logits_out=None, stream=None, timer=None):
        """Routing from the tokens themselves, in one launch: router GEMM
        (x W_r^T) with the top-k in its epilogue, then the same permutation
        as route(); w_router bf16 [E,d]; logits_out fp32 [T,E] or None."""
        self._x_row_fused = False
        with self._t(timer, "route_fused"):
            L.moe_route_permute_fused(self.desc, x, w_router, bias, logits_out, self.topk_idx,
                                      self.topk_w, self.counts, self.offsets,
                                      self.padded_offsets, self.tile_prefix, self.row_src,
                                      self.row_of, self.x_perm, self.ws, stream)

    def set_groups(self, counts, stream=None):
        """Groups given directly (no router): counts int32 [E] on device."""
        self.counts.copy_(counts)
        L.moe_group_offsets(self.desc, self.counts, self.offsets, self.padded_offsets,
                            self.tile_prefix, stream)

    def mx_buffers(self, width):
        """Device buffers for the optional MXFP8 / amax outputs of a tensor
        [capacity, width] (see moe_mx_out_t in include/moe.h)."""
        cap, dev, u8 = self.capacity, self.w2.device, torch.uint8
        return dict(q=torch.zeros((cap, width), dtype=u8, device=dev),
                    scale=torch.zeros((cap, width // 32), dtype=u8, device=dev),
                    qt=torch.zeros((width, cap), dtype=u8, device=dev),
                    scale_t=torch.zeros((width, cap // 32), dtype=u8, device=dev),
                    amax=torch.zeros(2, dtype=torch.float32, device=dev))

    def mlp_forward(self, stream=None, timer=None, a_mx=None, y_mx=None):
        c, po = self.counts, self.padded_offsets
        if self.f32:
            with self._t(timer, "transpose_x"):
                L.moe_transpose_rows_f32(self.desc, self.x_perm, self.d, po, self.x_t, stream)
            with self._t(timer, "fc1_glu_fwd"):
                L.moe_fc1_glu_fwd_tf32(self.desc, self.x_perm, c, po, self.w1p, self.b1p, self.h,
                                       self.a, self.a_t, stream)
            with self._t(timer, "fc2_fwd"):
                L.moe_fc2_fwd_tf32(self.desc, self.a, c, po, self.w2, self.b2, self.y, stream)
            return
        if a_mx is None and self.amax_a is not None and not self.mx:
            a_mx = dict(amax=self.amax_a)
        if self.nv:
            with self._t(timer, "quant_x"):
                L.moe_quantize_act_nvfp4(self.desc, self.x_perm, self.d, po, self.x_nv, True,
                                         stream)
            with self._t(timer, "fc1_glu_fwd"):
                L.moe_fc1_glu_fwd_nv(self.desc, self.x_nv, c, po, self.w_nv, self.b1p, self.h,
                                     self.a, self.a_nv["amax"], stream)
            with self._t(timer, "quant_a"):
                L.moe_quantize_act_nvfp4(self.desc, self.a, self.F, po, self.a_nv, False, stream)
            with self._t(timer, "fc2_fwd"):
                L.moe_fc2_fwd_nv(self.desc, self.a_nv, c, po, self.w_nv, self.b2, self.y, stream)
            return
        if self.mx:
            with self._t(timer, "quant_x"):
                L.moe_quantize_act_mx(self.desc, self.x_perm, self.d, po,
                                      self._colwise(self.x_mx) if self._x_row_fused else self.x_mx,
                                      stream)
            with self._t(timer, "fc1_glu_fwd"):
                a_out = self.a_mx if self.amax_a is None else dict(self.a_mx, amax=self.amax_a)
                L.moe_fc1_glu_fwd_mx(self.desc, self.x_mx, c, po, self.w_mx, self.b1p, self.h,
                                     self.a if self.keep_bf16 else None, a_out, stream)
            with self._t(timer, "fc2_fwd"):
                L.moe_fc2_fwd_mx(self.desc, self.a_mx, c, po, self.w_mx, self.b2, self.y, stream)
            return
        with self._t(timer, "fc1_glu_fwd"):
            L.moe_fc1_glu_fwd(self.desc, self.x_perm, c, po, self.w1p, self.b1p, self.h, self.a,
                              stream, mx=a_mx)
        with self._t(timer, "fc2_fwd"):
            L.moe_fc2_fwd(self.desc, self.a, c, po, self.w2, self.b2, self.y, stream, mx=y_mx)

    def mlp_backward(self, stream=None, timer=None, dh_mx=None):
        c, po = self.counts, self.padded_offsets
        if self.f32:
            with self._t(timer, "transpose_dy"):
                L.moe_transpose_rows_f32(self.desc, self.dy, self.d, po, self.dy_t, stream)
            with self._t(timer, "fc2_dgrad_dglu"):
                L.moe_fc2_dgrad_dglu_tf32(self.desc, self.dy, self.h, c, po, self.w2t, self.dh,
                                          self.dh_t, stream)
            with self._t(timer, "fc2_wgrad"):
                L.moe_fc2_wgrad_tf32(self.desc, self.dy_t, self.a_t, c, po, self.dw2, stream)
            with self._t(timer, "fc1_dgrad"):
                L.moe_fc1_dgrad_tf32(self.desc, self.dh, c, po, self.w1t, self.dx_perm, stream)
            with self._t(timer, "fc1_wgrad"):
                L.moe_fc1_wgrad_tf32(self.desc, self.dh_t, self.x_t, c, po, self.dw1p, stream)
            if self.has_b1 or self.has_b2:
                with self._t(timer, "bias_grads"):
                    L.moe_bias_grads(self.desc, self.dy, self.dh, c, po, self.db1p, self.db2,
                                     stream)
            return
        if dh_mx is None and self.amax_dh is not None and not self.mx:
            dh_mx = dict(amax=self.amax_dh)
        if self.nv:
            with self._t(timer, "quant_dy"):
                L.moe_quantize_act_nvfp4(self.desc, self.dy, self.d, po, self.dy_nv, True, stream)
            h = self.h
            if self.recompute_h:                  # regenerate H into a transient buffer
                h = torch.empty((self.capacity, self.W1), dtype=torch.bfloat16,
                                device=self.w2.device)
                with self._t(timer, "fc1_recompute_h"):
                    L.moe_fc1_recompute_h_nv(self.desc, self.x_nv, c, po, self.w_nv, self.b1p,
                                             h, stream)
            with self._t(timer, "fc2_dgrad_dglu"):
                L.moe_fc2_dgrad_dglu_nv(self.desc, self.dy_nv, h, c, po, self.w_nv, self.dh,
                                        self.dh_nv["amax"], stream)
            with self._t(timer, "quant_dh"):
                L.moe_quantize_act_nvfp4(self.desc, self.dh, self.W1, po, self.dh_nv, False,
                                         stream)
            with self._t(timer, "fc2_wgrad"):
                L.moe_fc2_wgrad_nv(self.desc, self.dy_nv, self.a_nv, c, po, self.dw2, stream)
            with self._t(timer, "fc1_dgrad"):
                L.moe_fc1_dgrad_nv(self.desc, self.dh_nv, c, po, self.w_nv, self.dx_perm, stream)
            with self._t(timer, "fc1_wgrad"):
                L.moe_fc1_wgrad_nv(self.desc, self.dh_nv, self.x_nv, c, po, self.dw1p, stream)
            if self.has_b1 or self.has_b2:
                with self._t(timer, "bias_grads"):
                    L.moe_bias_grads(self.desc, self.dy, self.dh, c, po, self.db1p, self.db2,
                                     stream)
            return
        if self.mx:
            with self._t(timer, "quant_dy"):
                L.moe_quantize_act_mx(self.desc, self.dy, self.d, po,
                                      self._colwise(self.dy_mx) if self._dy_row_fused
                                      else self.dy_mx, stream)
            dh_out = self.dh_mx if self.amax_dh is None else dict(self.dh_mx, amax=self.amax_dh)
            dh = self.dh if (self.keep_bf16 or self.has_b1) else None
            if self.recompute_h and self.gated:   # H recomputed inside the dGLU kernel
                with self._t(timer, "fc2_dgrad_dglu"):
                    L.moe_fc2_dgrad_dglu_recompute_mx(self.desc, self.x_mx, self.dy_mx, c, po,
                                                      self.w_mx, self.b1p, dh, dh_out, stream)
            else:
                h = self.h
                if self.recompute_h:              # regenerate H into a transient buffer
                    h = torch.empty((self.capacity, self.W1), dtype=torch.bfloat16,
                                    device=self.w2.device)
                    with self._t(timer, "fc1_recompute_h"):
                        L.moe_fc1_recompute_h_mx(self.desc, self.x_mx, c, po, self.w_mx,
                                                 self.b1p, h, stream)
                with self._t(timer, "fc2_dgrad_dglu"):
                    L.moe_fc2_dgrad_dglu_mx(self.desc, self.dy_mx, h, c, po, self.w_mx, dh,
                                            dh_out, stream)
            with self._t(timer, "fc2_wgrad"):
                L.moe_fc2_wgrad_mx(self.desc, self.dy_mx, self.a_mx, c, po, self.dw2, stream)
            with self._t(timer, "fc1_dgrad"):
                L.moe_fc1_dgrad_mx(self.desc, self.dh_mx, c, po, self.w_mx, self.dx_perm, stream)
            with self._t(timer, "fc1_wgrad"):
                L.moe_fc1_wgrad_mx(self.desc, self.dh_mx, self.x_mx, c, po, self.dw1p, stream)
            if self.has_b1 or self.has_b2:
                with self._t(timer, "bias_grads"):
                    L.moe_bias_grads(self.desc, self.dy, self.dh, c, po, self.db1p, self.db2,
                                     stream)
            return
        if self.recompute_h:
            with self._t(timer, "mlp_bwd_recompute"):
                L.moe_mlp_bwd(self.desc, self.dy, self.x_perm, None, self.a, c, po, self.w1p,
                              self.w2, self.dh, self.dx_perm, self.dw1p, self.db1p, self.dw2,
                              self.db2, self.ws, stream, dh_mx=dh_mx, b1p=self.b1p)
            return
        with self._t(timer, "fc2_dgrad_dglu"):
            L.moe_fc2_dgrad_dglu(self.desc, self.dy, self.h, c, po, self.w2, self.dh, stream,
                                 mx=dh_mx)
        with self._t(timer, "fc2_wgrad"):
            L.moe_fc2_wgrad(self.desc, self.dy, self.a, c, po, self.dw2, stream)
        with self._t(timer, "fc1_dgrad"):
            L.moe_fc1_dgrad(self.desc, self.dh, c, po, self.w1p, self.dx_perm, stream)
        with self._t(timer, "fc1_wgrad"):
            L.moe_fc1_wgrad(self.desc, self.dh, self.x_perm, c, po, self.dw1p, stream)
        if self.has_b1 or self.has_b2:
            with self._t(timer, "bias_grads"):
                L.moe_bias_grads(self.desc, self.dy, self.dh, c, po, self.db1p, self.db2, stream)

    # ---------------------------------------------------- unfused comparison
    # The arrangement the fused kernels replace: the group sizes read back to
    # the host each pass (one device-to-host copy and a synchronisation, as a
    # host-driven grouped GEMM needs them to size its launches), plain
    # grouped GEMMs, and the activation -- and on the MXFP8 path the
    # quantization of its output -- as separate memory-bound passes.
    def _host_sync_counts(self):
        self.host_counts = self.counts.cpu()

    def mlp_forward_unfused(self, stream=None, timer=None):
        """FC1 plain GEMM + separate GLU pass (+ separate MXFP8 quantization
        of A), then FC2."""
        c, po = self.counts, self.padded_offsets
        with self._t(timer, "host_sync"):
            self._host_sync_counts()
        if self.mx:
            with self._t(timer, "quant_x"):
                L.moe_quantize_act_mx(self.desc, self.x_perm, self.d, po, self.x_mx, stream)
            with self._t(timer, "fc1_glu_fwd"):
                L.moe_fc1_glu_fwd_mx_unfused(self.desc, self.x_mx, c, po, self.w_mx, self.b1p,
                                             self.h, self.a, self.a_mx, stream)
            with self._t(timer, "fc2_fwd"):
                L.moe_fc2_fwd_mx(self.desc, self.a_mx, c, po, self.w_mx, self.b2, self.y, stream)
            return
        with self._t(timer, "fc1_glu_fwd"):
            L.moe_fc1_glu_fwd_unfused(self.desc, self.x_perm, c, po, self.w1p, self.b1p, self.h,
                                      self.a, stream)
        with self._t(timer, "fc2_fwd"):
            L.moe_fc2_fwd(self.desc, self.a, c, po, self.w2, self.b2, self.y, stream)

    def mlp_backward_unfused(self, stream=None, timer=None):
        """FC2 dgrad plain GEMM + separate dGLU pass (+ separate MXFP8
        quantization of dH), then the weight gradients and FC1 dgrad."""
        if getattr(self, "da", None) is None:
            self.da = torch.zeros((self.capacity, self.F), dtype=torch.bfloat16,
                                  device=self.w2.device)
        c, po = self.counts, self.padded_offsets
        with self._t(timer, "host_sync"):
            self._host_sync_counts()
        if self.mx:
            with self._t(timer, "quant_dy"):
                L.moe_quantize_act_mx(self.desc, self.dy, self.d, po, self.dy_mx, stream)
            with self._t(timer, "fc2_dgrad_dglu"):
                L.moe_fc2_dgrad_dglu_mx_unfused(self.desc, self.dy_mx, self.h, c, po, self.w_mx,
                                                self.da, self.dh, self.dh_mx, stream)
            with self._t(timer, "fc2_wgrad"):
                L.moe_fc2_wgrad_mx(self.desc, self.dy_mx, self.a_mx, c, po, self.dw2, stream)
            with self._t(timer, "fc1_dgrad"):
                L.moe_fc1_dgrad_mx(self.desc, self.dh_mx, c, po, self.w_mx, self.dx_perm, stream)
            with self._t(timer, "fc1_wgrad"):
                L.moe_fc1_wgrad_mx(self.desc, self.dh_mx, self.x_mx, c, po, self.dw1p, stream)
        else:
            with self._t(timer, "fc2_dgrad_dglu"):
                L.moe_fc2_dgrad_dglu_unfused(self.desc, self.dy, self.h, c, po, self.w2, self.da,
                                             self.dh, stream)
            with self._t(timer, "fc2_wgrad"):
                L.moe_fc2_wgrad(self.desc, self.dy, self.a, c, po, self.dw2, stream)
            with self._t(timer, "fc1_dgrad"):
                L.moe_fc1_dgrad(self.desc, self.dh, c, po, self.w1p, self.dx_perm, stream)
            with self._t(timer, "fc1_wgrad"):
                L.moe_fc1_wgrad(self.desc, self.dh, self.x_perm, c, po, self.dw1p, stream)
        if self.has_b1 or self.has_b2:
            with self._t(timer, "bias_grads"):
                L.moe_bias_grads(self.desc, self.dy, self.dh, c, po, self.db1p, self.db2, stream)

    def forward(self, x, logits, bias=None, stream=None, timer=None):
        self.route(x, logits, bias, stream, timer)
        self.mlp_forward(stream, timer)
        with self._t(timer, "combine"):
            L.moe_unpermute_combine(self.desc, self.y, self.row_of, self.topk_w, self.out, stream)
        return self.out

    def backward(self, dout, stream=None, timer=None):
        with self._t(timer, "combine_bwd"):
            if self.mx:          # dY's rowwise MXFP8 copy written by the combine backward
                L.moe_unpermute_combine_bwd_mx(self.desc, dout, self.y, self.row_of, self.topk_w,
                                               self.row_src, self.padded_offsets, self.dy,
                                               self._rowwise(self.dy_mx), self.dw, stream)
                self._dy_row_fused = True
            else:
                L.moe_unpermute_combine_bwd(self.desc, dout, self.y, self.row_of, self.topk_w,
                                            self.row_src, self.padded_offsets, self.dy, self.dw,
                                            stream)
        self.mlp_backward(stream, timer)
        with self._t(timer, "permute_bwd"):
            L.moe_permute_bwd(self.desc, self.dx_perm, self.row_of, self.dx, stream)
        with self._t(timer, "route_bwd"):
            L.moe_route_bwd(self.desc, self.dw, self.topk_w, self.topk_idx, self.dlogits, stream)
        return self.dx

    def step(self, x, logits, bias, dout, stream=None, timer=None):
        """One whole forward + backward pass of the layer."""
        self.forward(x, logits, bias, stream, timer)
        self.backward(dout, stream, timer)

    def grouped_step(self, stream=None, timer=None, counts=None, x_perm=None, dy=None, y=None,
                     dx_perm=None):
        """Forward + backward of the expert MLP alone, for groups given
        directly (x_perm and dy already in place).  counts: new group sizes
        (int32 [E] on the device; the group offsets are recomputed on the
        device first).  x_perm, dy, y, dx_perm: [capacity, d] bf16 device
        tensors the layer reads its inputs from and writes its per-row
        results to from now on (no copy is made)."""
        self._x_row_fused = self._dy_row_fused = False   # x_perm, dy given directly
        if x_perm is not None:
            self.x_perm = x_perm
        if dy is not None:
            self.dy = dy
        if y is not None:
            self.y = y
        if dx_perm is not None:
            self.dx_perm = dx_perm
        if counts is not None:
            with self._t(timer, "group_offsets"):
                self.set_groups(counts, stream)
        self.mlp_forward(stream, timer)
        self.mlp_backward(stream, timer)

    def kernels_per_step(self, routed=True):
        """Kernels of this library launched by one step() (routed) or
        grouped_step(): six grouped GEMMs, one column-sum per bias, the two
        activation quantizations of the MXFP8 layer (NVFP4: four quantizations
        and two amax passes; fp32: the transposes of x_perm and dY), and for
        the routed layer top-k, group offsets + assignment (one launch),
        gather, combine, pad-row zeroing, combine backward, permute backward
        and router backward."""
        n = (6 + int(self.has_b1) + int(self.has_b2) + (2 if self.mx else 0) + (6 if self.nv else 0)
             + (2 if self.f32 else 0))
        return n + (8 if routed else 0)
