"""Device buffers for one decode step (PyTorch allocates, the library computes).

``DeviceStep`` holds device copies of a workload's inputs, the metadata outputs, the
split-K scratch and the outputs, and runs the three stages through the C ABI, either
one by one or as ``pa_decode_step``.  ``WindowStep`` adds the sliding-window pool of a
workload drawn with one and runs the sliding-window layer's step
(``pa_decode_step_window``).
"""

from __future__ import annotations

import torch

from . import binding as B


class DeviceStep:
    def __init__(self, wl, device="cuda", num_splits: int | None = None,
                 page_table_stride: int | None = None, with_swa: bool = True):
        spec = wl.spec
        self.spec = spec
        self.device = device
        self.bs = spec.bs
        self.num_q_heads, self.num_kv_heads = spec.num_q_heads, spec.num_kv_heads
        self.head_dim, self.page_size = spec.head_dim, spec.page_size
        self.seqlen_offset = spec.seqlen_offset
        self.max_seq_pages = wl.max_seq_pages
        self.sm_scale = wl.sm_scale
        to = dict(device=device)
        # q, req_pool_indices and seq_lens back to back in one buffer, out and lse in
        # another: the packed layout of pa_decode_step_host_packed (one copy each way)
        self._inputs = torch.empty(self._input_bytes(), dtype=torch.uint8, device=device)
        self.q, self.req_pool_indices, self.seq_lens = self._input_views(self._inputs)
        self.q.copy_(wl.q)
        self.req_pool_indices.copy_(wl.req_pool_indices)
        self.seq_lens.copy_(wl.seq_lens)
        self.req_to_token = wl.req_to_token.to(**to)
        # (a workload drawn without its full pool leaves these None)
        self.k_cache = wl.k_cache.to(**to) if wl.k_cache is not None else None
        self.v_cache = wl.v_cache.to(**to) if wl.v_cache is not None else None
        self.k_scale = wl.k_scale.to(**to) if wl.k_scale is not None else None
        self.v_scale = wl.v_scale.to(**to) if wl.v_scale is not None else None
        self.full_to_swa_mapping = (wl.full_to_swa_mapping.to(**to)
                                    if with_swa and wl.full_to_swa_mapping is not None else None)
        if num_splits is None:
            kv = B.PA_KV_INT8 if spec.kv_dtype == "int8" else B.PA_KV_BF16
            num_splits = spec.num_splits or B.pa_choose_splits(
                self.bs, self.num_kv_heads, self.max_seq_pages, self.page_size, kv)
        self.num_splits = int(num_splits)
        pts = page_table_stride or self.max_seq_pages
        i32 = dict(dtype=torch.int32, device=device)
        self.cache_seqlens = torch.empty(self.bs, **i32)
        self.cu_seqlens_k = torch.empty(self.bs + 1, **i32)
        self.page_table = torch.empty((self.bs, pts), **i32)
        self.swa_page_table = (torch.empty((self.bs, pts), **i32)
                               if self.full_to_swa_mapping is not None else None)
        f32 = dict(dtype=torch.float32, device=device)
        S = self.num_splits
        self.scratch_m = torch.empty((self.bs, self.num_q_heads, S), **f32)
        self.scratch_l = torch.empty((self.bs, self.num_q_heads, S), **f32)
        self.scratch_acc = torch.empty((self.bs, self.num_q_heads, S, self.head_dim), **f32)
        self.workspace = torch.empty(
            B.pa_workspace_bytes(self.bs, self.num_q_heads, self.head_dim, S),
            dtype=torch.uint8, device=device)
        self._outputs = torch.empty(self._output_bytes(), dtype=torch.uint8, device=device)
        self.out, self.lse = self._output_views(self._outputs)
        self._prepared = {}

    # ---- packed input / output groups ----------------------------------------------
    def _q_bytes(self):
        return self.bs * self.num_q_heads * self.head_dim * 2

    def _input_bytes(self):
        return self._q_bytes() + 2 * self.bs * 8

    def _output_bytes(self):
        return self._q_bytes() + self.bs * self.num_q_heads * 4

    def _input_views(self, buf):
        """q [bs, Hq, d] bf16, req_pool_indices [bs] int64, seq_lens [bs] int64, back to
        back in ``buf``."""
        qb = self._q_bytes()
        q = buf[:qb].view(torch.bfloat16).view(self.bs, self.num_q_heads, self.head_dim)
        rpi = buf[qb:qb + 8 * self.bs].view(torch.int64)
        sl = buf[qb + 8 * self.bs:qb + 16 * self.bs].view(torch.int64)
        return q, rpi, sl

    def _output_views(self, buf):
        """out [bs, Hq, d] bf16 and lse [bs, Hq] fp32, back to back in ``buf``."""
        qb = self._q_bytes()
        out = buf[:qb].view(torch.bfloat16).view(self.bs, self.num_q_heads, self.head_dim)
        lse = buf[qb:].view(torch.float32).view(self.bs, self.num_q_heads)
        return out, lse

    def host_buffers(self):
        """Pinned host buffers with the packed layout of pa_decode_step_host_packed:
        (h_inputs, h_outputs, views) with views = (h_q, h_req_pool_indices, h_seq_lens,
        h_out, h_lse) into them."""
        h_in = torch.empty(self._input_bytes(), dtype=torch.uint8, pin_memory=True)
        h_outs = torch.empty(self._output_bytes(), dtype=torch.uint8, pin_memory=True)
        return h_in, h_outs, (*self._input_views(h_in), *self._output_views(h_outs))

    def prepare_packed_host_step(self, h_inputs, h_outputs, use_pdl=True, stream=None):
        """A prepared ``pa_decode_step_host_packed`` call: h_inputs copied into this
        step's input group, the step, the output group copied to h_outputs."""
        return B.prepare_decode_step_host_packed(
            h_inputs=h_inputs, inputs=self._inputs, h_outputs=h_outputs,
            outputs=self._outputs, stream=B._stream(stream), use_pdl=use_pdl,
            **self._step_kwargs())

    # ---- the three stages ---------------------------------------------------------
    def metadata(self, use_pdl=True, stream=None):
        B.pa_build_metadata(self.req_pool_indices, self.seq_lens, self.req_to_token,
                            self.cache_seqlens, self.cu_seqlens_k, self.page_table,
                            seqlen_offset=self.seqlen_offset, max_seq_pages=self.max_seq_pages,
                            page_size=self.page_size, full_to_swa_mapping=self.full_to_swa_mapping,
                            swa_page_table=self.swa_page_table, stream=stream, use_pdl=use_pdl)

    def splitk(self, use_pdl=True, stream=None):
        B.pa_decode_splitk(self.q, self.k_cache, self.v_cache, self.page_table,
                           self.cache_seqlens, self.scratch_m, self.scratch_l, self.scratch_acc,
                           max_seq_pages=self.max_seq_pages, num_splits=self.num_splits,
                           sm_scale=self.sm_scale, k_scale=self.k_scale, v_scale=self.v_scale,
                           stream=stream, use_pdl=use_pdl)

    def reduce(self, use_pdl=True, stream=None):
        B.pa_reduce(self.scratch_m, self.scratch_l, self.scratch_acc, self.out, self.lse,
                    stream=stream, use_pdl=use_pdl)

    def stages(self, use_pdl=True, stream=None):
        self.metadata(use_pdl, stream)
        self.splitk(use_pdl, stream)
        self.reduce(use_pdl, stream)

    def _step_kwargs(self):
        return dict(req_pool_indices=self.req_pool_indices, seq_lens=self.seq_lens,
                    req_to_token=self.req_to_token, seqlen_offset=self.seqlen_offset,
                    max_seq_pages=self.max_seq_pages, cache_seqlens=self.cache_seqlens,
                    cu_seqlens_k=self.cu_seqlens_k, page_table=self.page_table, q=self.q,
                    k_cache=self.k_cache, v_cache=self.v_cache, num_splits=self.num_splits,
                    sm_scale=self.sm_scale, workspace=self.workspace, out=self.out,
                    lse=self.lse, k_scale=self.k_scale, v_scale=self.v_scale,
                    full_to_swa_mapping=self.full_to_swa_mapping,
                    swa_page_table=self.swa_page_table)

    _prepare = staticmethod(B.prepare_decode_step)

    def step(self, use_pdl=True, stream=None, lib=None):
        """One decode step through the C ABI.  The call is marshalled once per (stream,
        PDL, library) and reused: the buffers above must not be replaced afterwards (in
        place updates such as ``q.copy_`` are fine)."""
        key = (B._stream(stream), bool(use_pdl), id(lib))
        call = self._prepared.get(key)
        if call is None:
            call = self._prepare(lib=lib, stream=key[0], use_pdl=use_pdl, **self._step_kwargs())
            self._prepared[key] = call
        call()

    def prepare_host_io_step(self, h_inputs, h_outputs, use_pdl=True, stream=None):
        """A prepared step whose q, req_pool_indices and seq_lens (in ``h_inputs``) and
        out and lse (in ``h_outputs``) live in pinned host memory with the layout of
        ``host_buffers()``: the kernels read and write them over the host link, so the
        stream holds the three kernels and no copy."""
        q, rpi, sl = self._input_views(h_inputs)
        out, lse = self._output_views(h_outputs)
        kw = self._step_kwargs()
        kw.update(q=q, req_pool_indices=rpi, seq_lens=sl, out=out, lse=lse)
        return self._prepare(stream=B._stream(stream), use_pdl=use_pdl, **kw)

    def prepare_host_step(self, h_q, h_req_pool_indices, h_seq_lens, h_out, h_lse=None,
                          use_pdl=True, stream=None):
        """A prepared ``pa_decode_step_host`` call: host inputs copied into this step's
        q / req_pool_indices / seq_lens, the step, outputs copied to h_out / h_lse."""
        return B.prepare_decode_step_host(
            h_q=h_q, h_req_pool_indices=h_req_pool_indices, h_seq_lens=h_seq_lens, h_out=h_out,
            h_lse=h_lse, stream=B._stream(stream), use_pdl=use_pdl, **self._step_kwargs())

    # ---- accounting -----------------------------------------------------------------
    def kv_bytes(self, ctx) -> int:
        """Bytes of K and V (plus int8 scales) the step must read: every cached token of
        every request, for every KV head."""
        per_token = 2 * self.head_dim * self.k_cache.element_size()
        if self.k_scale is not None:
            per_token += 2 * 4
        return sum(ctx) * self.num_kv_heads * per_token

    def step_bytes(self, ctx) -> int:
        """Algorithmic HBM bytes of one decode step: KV (+scales), Q read, O and LSE
        written, split-K scratch written once and read once, and the metadata."""
        rows = self.bs * self.num_q_heads
        q_o = rows * self.head_dim * 2 * 2 + rows * 4
        scratch = 2 * rows * self.num_splits * (self.head_dim + 2) * 4
        meta = self.bs * (8 + 8 + 4 + 4) + 4 + self.bs * self.max_seq_pages * (4 + 4)
        if self.swa_page_table is not None:
            meta += self.bs * self.max_seq_pages * (4 + 8)
        return self.kv_bytes(ctx) + q_o + scratch + meta


class WindowStep(DeviceStep):
    """A sliding-window layer's decode step: the metadata stage, then the window
    producer over ``swa_page_table`` and the sliding-window pool, then the reducer."""

    def __init__(self, wl, device="cuda", num_splits: int | None = None):
        if wl.k_swa is None:
            raise ValueError("workload drawn without a sliding-window pool")
        spec = wl.spec
        self.window = int(spec.swa_window)
        if num_splits is None:
            pages = B.pa_window_pages(self.window, 1, spec.page_size, wl.max_seq_pages)
            kv = B.PA_KV_INT8 if spec.kv_dtype == "int8" else B.PA_KV_BF16
            num_splits = B.pa_choose_splits(spec.bs, spec.num_kv_heads, pages, spec.page_size, kv)
        super().__init__(wl, device=device, num_splits=num_splits, with_swa=True)
        to = dict(device=device)
        # the full pool is not read by this step: the sliding-window pool takes its place
        self.k_cache = wl.k_swa.to(**to)
        self.v_cache = wl.v_swa.to(**to)
        self.k_scale = wl.k_swa_scale.to(**to) if wl.k_swa_scale is not None else None
        self.v_scale = wl.v_swa_scale.to(**to) if wl.v_swa_scale is not None else None

    def splitk(self, use_pdl=True, stream=None):
        B.pa_decode_splitk_window(self.q, self.k_cache, self.v_cache, self.swa_page_table,
                                  self.cache_seqlens, self.scratch_m, self.scratch_l,
                                  self.scratch_acc, sliding_window=self.window,
                                  max_seq_pages=self.max_seq_pages, num_splits=self.num_splits,
                                  sm_scale=self.sm_scale, k_scale=self.k_scale,
                                  v_scale=self.v_scale, stream=stream, use_pdl=use_pdl)

    def _step_kwargs(self):
        return dict(req_pool_indices=self.req_pool_indices, seq_lens=self.seq_lens,
                    req_to_token=self.req_to_token, seqlen_offset=self.seqlen_offset,
                    max_seq_pages=self.max_seq_pages, cache_seqlens=self.cache_seqlens,
                    cu_seqlens_k=self.cu_seqlens_k, page_table=self.page_table,
                    full_to_swa_mapping=self.full_to_swa_mapping,
                    swa_page_table=self.swa_page_table, q=self.q, k_swa=self.k_cache,
                    v_swa=self.v_cache, sliding_window=self.window, num_splits=self.num_splits,
                    sm_scale=self.sm_scale, workspace=self.workspace, out=self.out,
                    lse=self.lse, k_swa_scale=self.k_scale, v_swa_scale=self.v_scale)

    _prepare = staticmethod(B.prepare_decode_step_window)

    def prepare_host_step(self, *args, **kwargs):
        raise NotImplementedError("host-buffer steps cover the full-attention layer only")

    def visible_tokens(self, ctx) -> list:
        """Positions each request's query attends: min(n, window)."""
        return [min(int(n), self.window) for n in ctx]

    def kv_bytes(self, ctx) -> int:
        """Bytes of K and V (plus int8 scales) the step must read: the window's tokens."""
        return super().kv_bytes(self.visible_tokens(ctx))
