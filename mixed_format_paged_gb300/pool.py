"""``MkvPool``: a pool whose device buffer is a torch tensor, with methods
that forward to the C ABI (``binding``).  Marshalling only."""
from __future__ import annotations

import torch

from . import binding as B


class MkvPool:
    def __init__(self, num_layers: int, num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 fp8_slots: int, tq3_slots: int, max_seqs: int, max_pages_per_seq: int, max_batch: int = 0,
                 rotation_seed: int = 0, device: str | torch.device = "cuda", host_only: bool = False,
                 stream=None):
        B.lib()   # raises when the CUDA library has not been built
        self.cfg = B.PoolConfig(num_layers, num_q_heads, num_kv_heads, head_dim, page_size, fp8_slots, tq3_slots,
                                max_seqs, max_pages_per_seq, max_batch, B.MKV_POOL_HOST_ONLY if host_only else 0,
                                0, rotation_seed)
        self.nbytes = B.mkv_pool_required_bytes(self.cfg)
        self.host_only = host_only
        self.buf = None
        if not host_only:
            self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
            if stream is None:
                stream = torch.cuda.current_stream(self.buf.device)
        self.handle = B.mkv_pool_create(self.cfg, self.buf, self.nbytes if self.buf is not None else 0, stream)
        self.head_dim = head_dim
        self.page_size = page_size
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads

    # ------------------------------------------------------------- lifetime
    def close(self) -> None:
        if self.handle is not None:
            B.mkv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream(self, stream):
        if stream is None and not self.host_only:
            return torch.cuda.current_stream(self.buf.device)
        return stream

    # ------------------------------------------------------------- forwarding
    def extend(self, seq_ids, n_new):
        B.mkv_seq_extend(self.handle, seq_ids, n_new)

    def release(self, seq: int):
        B.mkv_seq_release(self.handle, seq)

    def seq_info(self, seq: int):
        return B.mkv_seq_info(self.handle, seq)

    def page_info(self, seq: int, page: int):
        return B.mkv_page_info(self.handle, seq, page)

    def append(self, layer: int, seq_ids, n_new, k: torch.Tensor, v: torch.Tensor, stream=None):
        dtype = B.MKV_BF16 if k.dtype == torch.bfloat16 else B.MKV_F32
        if k.dtype != v.dtype or k.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("k and v must both be float32 or bfloat16")
        if not (k.is_contiguous() and v.is_contiguous()):
            raise ValueError("k and v must be contiguous")
        B.mkv_append_tokens(self.handle, layer, seq_ids, n_new, k, v, dtype, self._stream(stream))

    def set_tier(self, seq: int, page: int, tier: int):
        B.mkv_set_tier(self.handle, seq, page, tier)

    def demote(self, seq_ids, pages, stream=None):
        B.mkv_demote_pages(self.handle, seq_ids, pages, self._stream(stream))

    def decode(self, layer: int, seq_ids, q: torch.Tensor, out: torch.Tensor | None = None,
               lse: torch.Tensor | None = None, stream=None):
        n = len(seq_ids)
        if q.dtype not in (torch.bfloat16, torch.float32) or not q.is_contiguous():
            raise TypeError("q must be a contiguous float32 or bfloat16 tensor")
        if out is None:
            out = torch.empty((n, self.num_q_heads, self.head_dim), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((n, self.num_q_heads), dtype=torch.float32, device=q.device)
        dtype = B.MKV_BF16 if q.dtype == torch.bfloat16 else B.MKV_F32
        B.mkv_decode_attention(self.handle, layer, seq_ids, q, dtype, out, lse, self._stream(stream))
        return out, lse

    def decode_multi(self, layer: int, seq_ids, q: torch.Tensor, out: torch.Tensor | None = None,
                     lse: torch.Tensor | None = None, stream=None):
        """Attention of each request's last nq tokens (q: [n, nq, H_q, d]), query
        token i seeing the request's tokens up to its own position; returns
        out [n, nq, H_q, d] and lse [n, nq, H_q]."""
        n, nq = len(seq_ids), q.shape[1]
        if q.dtype not in (torch.bfloat16, torch.float32) or not q.is_contiguous() or q.dim() != 4:
            raise TypeError("q must be a contiguous [n, nq, H_q, d] float32 or bfloat16 tensor")
        if out is None:
            out = torch.empty((n, nq, self.num_q_heads, self.head_dim), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((n, nq, self.num_q_heads), dtype=torch.float32, device=q.device)
        dtype = B.MKV_BF16 if q.dtype == torch.bfloat16 else B.MKV_F32
        B.mkv_decode_attention_multi(self.handle, layer, seq_ids, nq, q, dtype, out, lse, self._stream(stream))
        return out, lse

    def append_decode(self, layer: int, seq_ids, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor,
                      out: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
        """Append each sequence's newest token (k, v: [n, H_kv, d]) and decode (q: [n, H_q, d])."""
        n = len(seq_ids)
        if out is None:
            out = torch.empty((n, self.num_q_heads, self.head_dim), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((n, self.num_q_heads), dtype=torch.float32, device=q.device)
        kvd = B.MKV_BF16 if k.dtype == torch.bfloat16 else B.MKV_F32
        qd = B.MKV_BF16 if q.dtype == torch.bfloat16 else B.MKV_F32
        B.mkv_append_decode(self.handle, layer, seq_ids, k, v, kvd, q, qd, out, lse, self._stream(stream))
        return out, lse

    def relevance(self, layer: int, seq_ids, q: torch.Tensor, lse: torch.Tensor, stream=None):
        """Attention mass per page ([n, max pages] fp32; zero past a sequence's
        pages) of the decode query q with that call's lse (mkv_page_relevance)."""
        n = len(seq_ids)
        npg = max(self.seq_info(r)[1] for r in seq_ids)
        mass = torch.zeros((n, npg), dtype=torch.float32, device=q.device)
        qd = B.MKV_BF16 if q.dtype == torch.bfloat16 else B.MKV_F32
        B.mkv_page_relevance(self.handle, layer, seq_ids, q, qd, lse, mass, npg, self._stream(stream))
        return mass

    def step_graph(self, seq_ids, q, out, lse, k=None, v=None, stream=None):
        """Record one decode step over every layer as a CUDA graph on fixed
        buffers (lists with one tensor per layer; k = v = None: no fused
        append).  Returns a StepGraph; its launch() runs one step."""
        qd = B.MKV_BF16 if q[0].dtype == torch.bfloat16 else B.MKV_F32
        kvd = B.MKV_BF16 if (k is not None and k[0].dtype == torch.bfloat16) else B.MKV_F32
        g = B.mkv_step_graph_create(self.handle, seq_ids, q, k, v, qd, kvd, out, lse, self._stream(stream))
        return StepGraph(self, g, (q, k, v, out, lse))

    def dequantize(self, layer: int, seq: int, page0: int, npages: int, dtype=torch.float32, stream=None):
        """Dense K, V [npages * P, H_kv, d] of pages [page0, page0 + npages)."""
        shape = (npages * self.page_size, self.num_kv_heads, self.head_dim)
        k = torch.empty(shape, dtype=dtype, device=self.buf.device)
        v = torch.empty(shape, dtype=dtype, device=self.buf.device)
        od = B.MKV_BF16 if dtype == torch.bfloat16 else B.MKV_F32
        B.mkv_dequantize_pages(self.handle, layer, seq, page0, npages, k, v, od, self._stream(stream))
        return k, v

    def stats(self):
        return B.mkv_pool_stats(self.handle)

    def export_page(self, layer: int, seq: int, page: int, stream=None):
        tier, _ = self.page_info(seq, page)
        P, H, D = self.page_size, self.num_kv_heads, self.head_dim
        nbytes = H * 2 * P * ((3 * D // 8 if tier == B.MKV_TIER_STALE else D) + 2)
        return B.mkv_export_page(self.handle, layer, seq, page, nbytes, self._stream(stream))

    def rotation_signs(self):
        return B.mkv_rotation_signs(self.handle, self.head_dim)

    def plan(self, seq_ids, nq: int = 1):
        if nq == 1:
            return B.mkv_plan_decode(self.handle, seq_ids)
        return B.mkv_plan_decode_multi(self.handle, seq_ids, nq)

    def check_device_errors(self, stream=None):
        B.mkv_check_device_errors(self.handle, self._stream(stream))

    def selftest_wait_timeout(self, limit_cycles: int = 2_000_000, stream=None):
        """Enqueue a bounded wait that runs out (see mkv_selftest_wait_timeout)."""
        B.mkv_selftest_wait_timeout(self.handle, limit_cycles, self._stream(stream))


class StepGraph:
    """A recorded decode step (mkv_step_graph_*); keeps its buffers alive."""

    def __init__(self, pool, handle, buffers):
        self.pool = pool
        self.handle = handle
        self.buffers = buffers

    def launch(self, stream=None):
        B.mkv_step_graph_launch(self.handle, self.pool._stream(stream))

    def close(self):
        if self.handle is not None:
            B.mkv_step_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
