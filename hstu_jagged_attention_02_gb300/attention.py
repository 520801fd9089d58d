"""Torch-facing helpers around the C ABI: device buffers for one jagged batch,
and an autograd function.  Marshalling only; the arithmetic is in the CUDA
kernels of libhstu_attn.so."""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import binding as C


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_handle(stream: Optional[torch.cuda.Stream] = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def torch_dtype(name: str):
    return torch.bfloat16 if name == "bf16" else torch.float32


class Problem:
    """Device copies of one synth.Batch plus every output buffer and the
    workspace, with the C argument structs filled once."""

    def __init__(self, batch, device="cuda", flags: int = 0, want_y: bool = True,
                 want_stats: bool = False, want_drab: bool = True, out_dtype: str = "fp32",
                 dropout=None, bwd_flags: int = 0, plan_once: bool = False, packed_inputs: bool = False):
        # dropout: None or (p, seed, offset) of the fused dropout on y;
        # bwd_flags: flags added for the backward call only (e.g.
        # HSTU_FLAG_FORCE_SIMT for a BF16 backward without a tensor-core kernel);
        # plan_once: the forward plans the backward too (HSTU_FLAG_PLAN_BWD)
        # and the backward reuses that plan (HSTU_FLAG_REUSE_PLAN);
        # packed_inputs: every input lives in one device buffer
        # (self.input_buffer, 256-byte aligned slots), so a host copy of the
        # whole batch is one transfer
        self.batch = batch
        dev = torch.device(device)
        self.dev = dev
        td = torch_dtype(batch.dtype)
        self.td = td
        out_dtype = "fp32" if batch.dtype == "fp32" else out_dtype
        self.out_dtype = out_dtype
        to = torch_dtype(out_dtype)
        self.to = to
        T, H, dqk, dv = batch.T, batch.H, batch.d_qk, batch.d_v
        F = H * dv
        self.T, self.H, self.F = T, H, F

        def up(a, dt=None):
            if a is None:
                return None
            t = torch.from_numpy(np.ascontiguousarray(a))
            return t.to(device=dev, dtype=dt if dt is not None else t.dtype)

        self.offsets = up(batch.offsets, torch.int64)
        self.num_targets = up(batch.num_targets, torch.int32)
        self.num_contexts = up(batch.num_contexts, torch.int32)
        self.timestamps = up(batch.timestamps, torch.int64)
        self.rab_pos = up(batch.rab_pos, torch.float32)
        self.rab_time = up(batch.rab_time, torch.float32)
        self.q, self.k, self.v = up(batch.q, td), up(batch.k, td), up(batch.v, td)
        self.u = up(batch.u, torch.float32 if flags & C.HSTU_FLAG_U_FP32 else td)
        self.dy = up(batch.dy, to)
        self.input_buffer = None
        if packed_inputs:
            self._pack_inputs()
        z = lambda *s, dt=to: torch.empty(*s, device=dev, dtype=dt)
        self.o = z(T, H, dv)
        self.y = z(T, F) if want_y else None
        self.mean = z(T, dt=torch.float32) if want_stats else None
        self.rstd = z(T, dt=torch.float32) if want_stats else None
        self.backward_enabled = batch.dy is not None
        if self.backward_enabled:
            self.dq, self.dk, self.dvv = z(T, H, dqk), z(T, H, dqk), z(T, H, dv)
            self.du = z(T, F) if self.u is not None else None
            self.d_rab_pos = (z(H, self.rab_pos.shape[1], dt=torch.float32)
                              if (self.rab_pos is not None and want_drab) else None)
            self.d_rab_time = (z(H, self.rab_time.shape[1], dt=torch.float32)
                               if (self.rab_time is not None and want_drab) else None)
        self.desc = C.make_desc(
            dtype=batch.dtype, out_dtype=out_dtype, B=batch.B, H=H, d_qk=dqk, d_v=dv, total_tokens=T,
            max_seq_len=batch.max_seq_len, alpha=batch.alpha,
            num_pos_buckets=batch.rab_pos.shape[1] if batch.rab_pos is not None else 128,
            num_time_buckets=batch.rab_time.shape[1] if batch.rab_time is not None else 64,
            norm=batch.norm, ln_eps=batch.eps, flags=flags,
            dropout_p=0.0 if dropout is None else float(dropout[0]))
        self.bwd_flags = bwd_flags
        self.plan_once = plan_once and batch.dy is not None
        if self.plan_once:
            self.bwd_flags |= C.HSTU_FLAG_REUSE_PLAN
        seed, offset = (0, 0) if dropout is None else (int(dropout[1]), int(dropout[2]))
        fwd_b, bwd_b = C.hstu_attn_workspace_size(self.desc)
        self.ws_bytes = max(fwd_b, bwd_b if self.backward_enabled else 0)
        self.ws = torch.empty(self.ws_bytes, device=dev, dtype=torch.uint8)
        self.fwd_args = C.hstu_attn_fwd_args(
            _ptr(self.offsets), _ptr(self.num_targets), _ptr(self.num_contexts), _ptr(self.timestamps),
            _ptr(self.rab_pos), _ptr(self.rab_time), _ptr(self.q), _ptr(self.k), _ptr(self.v),
            _ptr(self.u), _ptr(self.o), _ptr(self.y), _ptr(self.mean), _ptr(self.rstd), seed, offset)
        if self.backward_enabled:
            self.bwd_args = C.hstu_attn_bwd_args(
                _ptr(self.offsets), _ptr(self.num_targets), _ptr(self.num_contexts),
                _ptr(self.timestamps), _ptr(self.rab_pos), _ptr(self.rab_time), _ptr(self.q),
                _ptr(self.k), _ptr(self.v), _ptr(self.u), _ptr(self.o), _ptr(self.dy),
                _ptr(self.dq), _ptr(self.dk), _ptr(self.dvv), _ptr(self.du), _ptr(self.d_rab_pos),
                _ptr(self.d_rab_time), seed, offset)

    _INPUTS = ("offsets", "num_targets", "num_contexts", "timestamps", "rab_pos", "rab_time", "q", "k", "v",
               "u", "dy")

    def _pack_inputs(self):
        """Move every input tensor into one device buffer (views at 256-byte
        aligned offsets)."""
        names = [n for n in self._INPUTS if getattr(self, n) is not None]
        offs, total = {}, 0
        for n in names:
            t = getattr(self, n)
            offs[n] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(max(total, 256), device=self.dev, dtype=torch.uint8)
        for n in names:
            t = getattr(self, n)
            nbytes = t.numel() * t.element_size()
            view = buf[offs[n]:offs[n] + nbytes].view(t.dtype).view(t.shape)
            view.copy_(t)
            setattr(self, n, view)
        self.input_buffer = buf

    def forward(self, stream=None):
        d = self.desc
        if self.plan_once:
            d = C.hstu_attn_desc.from_buffer_copy(self.desc)
            d.flags |= C.HSTU_FLAG_PLAN_BWD
        C.hstu_attn_fwd(d, self.fwd_args, self.ws.data_ptr(), self.ws_bytes, _stream_handle(stream))

    def backward(self, stream=None):
        d = C.hstu_attn_desc.from_buffer_copy(self.desc)
        d.flags |= self.bwd_flags
        C.hstu_attn_bwd(d, self.bwd_args, self.ws.data_ptr(), self.ws_bytes, _stream_handle(stream))

    def device_error(self, stream=None) -> int:
        return C.hstu_get_device_error(self.ws.data_ptr(), _stream_handle(stream))

    def debug_plan(self, pass_: int, capacity: int, stream=None):
        need = self.ws_bytes + 24 * capacity + 512
        ws = torch.empty(need, device=self.dev, dtype=torch.uint8)
        return C.hstu_attn_debug_plan(self.desc, _ptr(self.offsets), _ptr(self.num_targets),
                                      _ptr(self.num_contexts), pass_, ws.data_ptr(), need, capacity,
                                      _stream_handle(stream))


class HSTUAttnFunction(torch.autograd.Function):
    """y = Norm(A V) * u with A = SiLU(alpha Q K^T + rab) / N under the
    compound mask; gradients for q, k, v, u, rab_pos, rab_time.

    The library computes o, y and every gradient in out_dtype ("fp32", the
    default, or "bf16"; FP32 inputs always give FP32).  An FP32 u with BF16
    q, k, v is read as FP32 (HSTU_FLAG_U_FP32).  Autograd hands each gradient
    back in the dtype of its input, so BF16 q, k, v receive the FP32 results
    rounded once to BF16."""

    @staticmethod
    def forward(ctx, q, k, v, u, rab_pos, rab_time, seq_offsets, num_targets, num_contexts,
                timestamps, max_seq_len: int, alpha: float, norm: str = "layernorm",
                eps: float = 1e-5, dropout_p: float = 0.0, dropout_seed: int = 0, dropout_offset: int = 0,
                out_dtype: Optional[str] = None, flags: int = 0):
        T, H, dqk = q.shape
        dv = v.shape[2]
        dtype = "bf16" if q.dtype == torch.bfloat16 else "fp32"
        out_dtype = "fp32" if (dtype == "fp32" or out_dtype is None) else out_dtype
        if dtype == "bf16" and u is not None and u.dtype == torch.float32:
            flags |= C.HSTU_FLAG_U_FP32
        to = torch_dtype(out_dtype)
        desc = C.make_desc(dtype=dtype, out_dtype=out_dtype, B=seq_offsets.numel() - 1, H=H, d_qk=dqk, d_v=dv,
                           total_tokens=T, max_seq_len=max_seq_len, alpha=alpha,
                           num_pos_buckets=rab_pos.shape[1] if rab_pos is not None else 128,
                           num_time_buckets=rab_time.shape[1] if rab_time is not None else 64,
                           norm=norm, ln_eps=eps, flags=flags, dropout_p=dropout_p)
        fwd_b, bwd_b = C.hstu_attn_workspace_size(desc)
        ws = torch.empty(max(fwd_b, bwd_b), device=q.device, dtype=torch.uint8)
        o = torch.empty(T, H, dv, device=q.device, dtype=to)
        y = torch.empty(T, H * dv, device=q.device, dtype=to)
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        u = u.contiguous() if u is not None else None
        args = C.hstu_attn_fwd_args(_ptr(seq_offsets), _ptr(num_targets), _ptr(num_contexts),
                                    _ptr(timestamps), _ptr(rab_pos), _ptr(rab_time), _ptr(q), _ptr(k),
                                    _ptr(v), _ptr(u), _ptr(o), _ptr(y), None, None, dropout_seed,
                                    dropout_offset)
        C.hstu_attn_fwd(desc, args, ws.data_ptr(), ws.numel(), _stream_handle())
        ctx.save_for_backward(q, k, v, u, rab_pos, rab_time, seq_offsets, num_targets, num_contexts,
                              timestamps, o)
        ctx.desc, ctx.ws, ctx.drop, ctx.to = desc, ws, (dropout_seed, dropout_offset), to
        return y

    @staticmethod
    def backward(ctx, dy):
        q, k, v, u, rab_pos, rab_time, off, nt, nc, ts, o = ctx.saved_tensors
        to = ctx.to
        dy = dy.contiguous().to(to)
        dq = torch.empty(q.shape, device=q.device, dtype=to)
        dk = torch.empty(k.shape, device=k.device, dtype=to)
        dv = torch.empty(v.shape, device=v.device, dtype=to)
        du = torch.empty(u.shape, device=u.device, dtype=to) if u is not None else None
        drp = torch.empty_like(rab_pos, dtype=torch.float32) if rab_pos is not None else None
        drt = torch.empty_like(rab_time, dtype=torch.float32) if rab_time is not None else None
        args = C.hstu_attn_bwd_args(_ptr(off), _ptr(nt), _ptr(nc), _ptr(ts), _ptr(rab_pos), _ptr(rab_time),
                                    _ptr(q), _ptr(k), _ptr(v), _ptr(u), _ptr(o), _ptr(dy), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(du), _ptr(drp), _ptr(drt), *ctx.drop)
        C.hstu_attn_bwd(ctx.desc, args, ctx.ws.data_ptr(), ctx.ws.numel(), _stream_handle())
        return (dq, dk, dv, du, drp, drt) + (None,) * 13


def hstu_attention(q, k, v, u, seq_offsets, max_seq_len, alpha, *, num_targets=None, num_contexts=None,
                   timestamps=None, rab_pos=None, rab_time=None, norm="layernorm", eps=1e-5,
                   dropout_p=0.0, dropout_seed=0, dropout_offset=0, out_dtype=None, flags=0):
    """Differentiable HSTU jagged attention: returns y [T, H*d_v] (with the
    fused dropout when dropout_p > 0; the seed and offset select the mask).
    out_dtype: "fp32" (default) or "bf16" for o, y and the library's
    gradients; flags: HSTU_FLAG_* bits (e.g. HSTU_FLAG_FORCE_SIMT)."""
    return HSTUAttnFunction.apply(q, k, v, u, rab_pos, rab_time, seq_offsets, num_targets, num_contexts,
                                  timestamps, int(max_seq_len), float(alpha), norm, float(eps),
                                  float(dropout_p), int(dropout_seed), int(dropout_offset), out_dtype, int(flags))
