"""Buffers and launch for one decode problem, through the C ABI.

``Decoder`` sizes the workspace and semaphores with the library's own queries,
allocates them (zeroed) with torch once, and launches ``xqa_decode`` or
``xqa_mla_decode`` on every ``run()``.
"""

from __future__ import annotations

import torch

from . import xqa as X


class Decoder:
    def __init__(self, case, sm_count=None, error_word=True, lse=False, out_dtype=None):
        if not case.q.is_cuda:
            raise ValueError("Decoder needs the problem on a CUDA device")
        self.case = case
        dev = case.q.device
        B, qs, Hq, _ = case.q.shape
        # the output takes the query's dtype; an e4m3 query (MLA with an e4m3
        # latent cache) writes bf16
        default_out = torch.bfloat16 if case.q.dtype == torch.float8_e4m3fn else case.q.dtype
        self.output = torch.empty((B, qs, Hq, case.dv), dtype=out_dtype or default_out, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev) if error_word else None
        self.lse = torch.empty((B, qs, Hq), dtype=torch.float32, device=dev) if lse else None
        kw = case.kwargs()
        v_head_dim = kw.pop("v_head_dim")
        self.params = X.make_params(case.q, case.k_cache, case.v_cache, case.page_table,
                                    case.seq_lens, self.output, q_seq_len=qs, sm_count=sm_count,
                                    error_word=self.err, lse=self.lse, **kw)
        self.mla = case.mla
        self.v_head_dim = case.dv
        if self.mla:
            ws = X.xqa_mla_workspace_size(self.params, self.v_head_dim)
            ns = X.xqa_mla_semaphore_count(self.params, self.v_head_dim)
        else:
            ws = X.xqa_workspace_size(self.params)
            ns = X.xqa_semaphore_count(self.params)
        self.workspace = torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev)
        # kernel launches per call: the latent decode adds its split merge
        # kernel whenever it needs a workspace
        self.launches_per_call = 2 if (self.mla and ws > 0) else 1
        self.semaphores = torch.zeros(max(ns, 1), dtype=torch.int32, device=dev)

    def run(self, stream=None):
        # (the semaphores were sized by the library's query at construction)
        if self.mla:
            X.xqa_mla_decode(self.params, self.v_head_dim, self.workspace, self.semaphores, stream,
                             check_semaphores=False)
        else:
            X.xqa_decode(self.params, self.workspace, self.semaphores, stream, check_semaphores=False)
        return self.output

    def error_bits(self):
        return 0 if self.err is None else int(self.err.item())
