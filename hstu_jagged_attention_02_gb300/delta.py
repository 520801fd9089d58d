"""Device buffers for the delta forward (KV-cached, candidate-only inference)
through hstu_attn_fwd_delta of libhstu_attn.so.  Marshalling only.

A jagged batch whose sequences end in m_b candidates is split into the cached
part (the first L_b = n_b - m_b tokens of each sequence: their K, V and
timestamps) and the candidates (their q, k, v, u and timestamps).  The delta
call then computes the candidates' o and y, which equal the candidate rows of
the full forward."""
from __future__ import annotations

import numpy as np
import torch

from . import binding as C
from .attention import _ptr, _stream_handle, torch_dtype


def split_rows(batch):
    """(cached-row indices, candidate-row indices, cache offsets, candidate
    offsets) of a jagged batch, in token order."""
    off = batch.offsets.astype(np.int64)
    m = batch.num_targets.astype(np.int64) if batch.num_targets is not None else np.zeros(batch.B, np.int64)
    cache_rows, cand_rows = [], []
    for b in range(batch.B):
        h_end = int(off[b + 1] - m[b])
        cache_rows.append(np.arange(off[b], h_end))
        cand_rows.append(np.arange(h_end, off[b + 1]))
    cache_rows = np.concatenate(cache_rows) if cache_rows else np.zeros(0, np.int64)
    cand_rows = np.concatenate(cand_rows) if cand_rows else np.zeros(0, np.int64)
    lens = off[1:] - off[:-1]
    cache_off = np.concatenate([[0], np.cumsum(lens - m)]).astype(np.int64)
    cand_off = np.concatenate([[0], np.cumsum(m)]).astype(np.int64)
    return cache_rows, cand_rows, cache_off, cand_off


class DeltaProblem:
    """Cached K/V and candidate tensors of one batch on the device, outputs
    and workspace, with the C argument struct filled once."""

    def __init__(self, batch, device="cuda", flags: int = 0, out_dtype: str = "fp32"):
        self.batch = batch
        dev = torch.device(device)
        td, to = torch_dtype(batch.dtype), torch_dtype(out_dtype)
        cache_rows, cand_rows, cache_off, cand_off = split_rows(batch)
        self.cache_rows, self.cand_rows = cache_rows, cand_rows
        H, d = batch.H, batch.d_v
        Tc, Tk = len(cand_rows), len(cache_rows)
        self.T_cand, self.T_cache = Tc, Tk

        def up(a, dt):
            if a is None:
                return None
            return torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)

        self.cand_offsets = up(cand_off, torch.int64)
        self.cache_offsets = up(cache_off, torch.int64)
        ts = batch.timestamps
        self.cand_ts = up(ts[cand_rows], torch.int64) if ts is not None else None
        self.cache_ts = up(ts[cache_rows], torch.int64) if ts is not None else None
        self.rab_pos = up(batch.rab_pos, torch.float32)
        self.rab_time = up(batch.rab_time, torch.float32)
        self.q, self.k, self.v = (up(x[cand_rows], td) for x in (batch.q, batch.k, batch.v))
        self.u = up(batch.u[cand_rows], torch.float32 if flags & C.HSTU_FLAG_U_FP32 else td) \
            if batch.u is not None else None
        self.k_cache, self.v_cache = up(batch.k[cache_rows], td), up(batch.v[cache_rows], td)
        self.o = torch.empty(Tc, H, d, device=dev, dtype=to)
        self.y = torch.empty(Tc, H * d, device=dev, dtype=to)
        self.desc = C.make_desc(
            dtype=batch.dtype, out_dtype=out_dtype, B=batch.B, H=H, d_qk=batch.d_qk, d_v=d, total_tokens=Tc,
            max_seq_len=batch.max_seq_len, alpha=batch.alpha,
            num_pos_buckets=batch.rab_pos.shape[1] if batch.rab_pos is not None else 128,
            num_time_buckets=batch.rab_time.shape[1] if batch.rab_time is not None else 64,
            norm=batch.norm, ln_eps=batch.eps, flags=flags)
        self.ws_bytes, _ = C.hstu_attn_workspace_size(self.desc)
        self.ws = torch.empty(self.ws_bytes, device=dev, dtype=torch.uint8)
        self.args = C.hstu_attn_delta_args(
            _ptr(self.cand_offsets), _ptr(self.cache_offsets), Tk, _ptr(self.cand_ts), _ptr(self.cache_ts),
            _ptr(self.rab_pos), _ptr(self.rab_time), _ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.u),
            _ptr(self.k_cache), _ptr(self.v_cache), _ptr(self.o), _ptr(self.y), None, None)

    def forward(self, stream=None):
        C.hstu_attn_fwd_delta(self.desc, self.args, self.ws.data_ptr(), self.ws_bytes, _stream_handle(stream))

    def device_error(self, stream=None) -> int:
        return C.hstu_get_device_error(self.ws.data_ptr(), _stream_handle(stream))
