"""Device buffers for one full HSTU layer (x W1 -> SiLU -> U, V, Q, K ->
attention -> y W2 + x) and its backward, through hstu_layer_fwd /
hstu_layer_bwd of libhstu_attn.so.  Marshalling only."""
from __future__ import annotations

import numpy as np
import torch

from . import binding as C
from .attention import _ptr, _stream_handle


class LayerProblem:
    """Device copies of a synth.layer batch (x, w1, w2, dout, offsets,
    timestamps, bias tables) plus every output and the workspace."""

    def __init__(self, batch, device="cuda", want_drab: bool = True, dropout=None, bwd_flags: int = 0):
        # dropout: None or (p, seed, offset) of the fused dropout on y;
        # bwd_flags: flags added for the backward call only (HSTU_FLAG_FORCE_SIMT
        # runs an attention backward without a tensor-core kernel, d != 128)
        self.batch = batch
        dev = torch.device(device)
        self.dev = dev
        T, H, d = batch.T, batch.H, batch.d_v
        D = H * d
        self.T, self.D = T, D

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
        self.x = up(batch.x, torch.bfloat16)
        self.w1 = up(batch.w1, torch.bfloat16)
        self.w2 = up(batch.w2, torch.bfloat16)
        self.dout = up(batch.dout, torch.float32) if batch.dout is not None else None
        f32 = dict(device=dev, dtype=torch.float32)
        self.out = torch.empty(T, D, **f32)
        self.z1 = torch.empty(T, 4 * D, **f32)
        self.u = torch.empty(T, D, **f32)
        self.vqk = torch.empty(3, T, D, device=dev, dtype=torch.bfloat16)
        self.o = torch.empty(T, D, **f32)
        self.y = torch.empty(T, D, **f32)
        self.backward_enabled = self.dout is not None
        if self.backward_enabled:
            self.dx = torch.empty(T, D, **f32)
            self.dw1 = torch.empty(D, 4 * D, **f32)
            self.dw2 = torch.empty(D, D, **f32)
            self.d_rab_pos = (torch.empty(H, self.rab_pos.shape[1], **f32)
                              if (self.rab_pos is not None and want_drab) else None)
            self.d_rab_time = (torch.empty(H, self.rab_time.shape[1], **f32)
                               if (self.rab_time is not None and want_drab) else None)
        self.desc = C.make_desc(
            dtype="bf16", out_dtype="fp32", B=batch.B, H=H, d_qk=batch.d_qk, d_v=d, total_tokens=T,
            max_seq_len=batch.max_seq_len, alpha=batch.alpha,
            num_pos_buckets=batch.rab_pos.shape[1] if batch.rab_pos is not None else 128,
            num_time_buckets=batch.rab_time.shape[1] if batch.rab_time is not None else 64,
            norm=batch.norm, ln_eps=batch.eps, dropout_p=0.0 if dropout is None else float(dropout[0]))
        self.bwd_flags = bwd_flags
        drop = (0, 0) if dropout is None else (int(dropout[1]), int(dropout[2]))
        fwd_b, bwd_b = C.hstu_layer_workspace_size(self.desc)
        self.ws_bytes = max(fwd_b, bwd_b if self.backward_enabled else 0)
        self.ws = torch.empty(self.ws_bytes, device=dev, dtype=torch.uint8)
        common = (_ptr(self.offsets), _ptr(self.num_targets), _ptr(self.num_contexts), _ptr(self.timestamps),
                  _ptr(self.rab_pos), _ptr(self.rab_time), _ptr(self.x), _ptr(self.w1), _ptr(self.w2))
        self.fwd_args = C.hstu_layer_fwd_args(*common, _ptr(self.out), _ptr(self.z1), _ptr(self.u),
                                              _ptr(self.vqk), _ptr(self.o), _ptr(self.y), *drop)
        if self.backward_enabled:
            self.bwd_args = C.hstu_layer_bwd_args(
                *common, _ptr(self.z1), _ptr(self.u), _ptr(self.vqk), _ptr(self.o), _ptr(self.y), _ptr(self.dout),
                _ptr(self.dx), _ptr(self.dw1), _ptr(self.dw2), _ptr(self.d_rab_pos), _ptr(self.d_rab_time),
                *drop)

    def forward(self, stream=None):
        C.hstu_layer_fwd(self.desc, self.fwd_args, self.ws.data_ptr(), self.ws_bytes, _stream_handle(stream))

    def backward(self, stream=None):
        d = C.hstu_attn_desc.from_buffer_copy(self.desc)
        d.flags |= self.bwd_flags
        C.hstu_layer_bwd(d, self.bwd_args, self.ws.data_ptr(), self.ws_bytes, _stream_handle(stream))

    def device_error(self, stream=None) -> int:
        return C.hstu_get_device_error(self.ws.data_ptr(), _stream_handle(stream))
