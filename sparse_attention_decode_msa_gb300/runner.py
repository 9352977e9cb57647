"""Device-side plumbing: put a synthetic problem in HBM and call the C ABI.

PyTorch is used only to allocate device memory and to provide the stream;
every computation runs in the library's kernels.
"""

from __future__ import annotations

import numpy as np

from . import (make_shape, msa_decode_step, msa_index_score, msa_kv_update, msa_select_topk,
               msa_sparse_decode, msa_workspace_bytes, msa_workspace_init)


def _dev(a, device):
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


class DeviceProblem:
    """A synthetic problem resident on one GPU, with output and workspace buffers."""

    def __init__(self, pb, device="cuda", decode_ctas: int = 0):
        import torch

        self.pb = pb
        self.device = device
        self.shape = make_shape(
            num_requests=pb.num_requests, q_per_req=pb.q_per_req, num_kv_heads=pb.num_kv_heads,
            num_pages=pb.num_pages, max_blocks_per_seq=pb.max_blocks, topk=pb.topk,
            kv_dtype=pb.kv_dtype, index_dtype=pb.index_dtype, softmax_scale=pb.softmax_scale,
            k_scale=pb.k_scale, v_scale=pb.v_scale, decode_ctas=decode_ctas,
            num_index_heads=getattr(pb, "num_index_heads", 1),
            init_blocks=getattr(pb, "init_blocks", 0), local_blocks=getattr(pb, "local_blocks", 0))
        self.q_idx = _dev(pb.q_idx, device)
        self.idxk = _dev(pb.idxk_pool, device)
        self.idxk_scales = None if pb.idxk_scales is None else _dev(pb.idxk_scales, device)
        self.q = _dev(pb.q, device)
        self.kv = _dev(pb.kv_pool, device)
        self.block_table = _dev(pb.block_table, device)
        self.seq_lens = _dev(pb.seq_lens, device)
        T, Hq = pb.num_tokens, pb.num_q_heads
        Hi = self.shape.num_index_heads
        Hs = 1 if Hi == 1 else pb.num_kv_heads      # selection tables per token
        self.block_scores = torch.full((T, Hi, pb.max_blocks), float("nan"), device=device)
        self.selected = torch.full((T, Hs, pb.topk), -7, dtype=torch.int32, device=device)
        self.out = torch.full((T, Hq, 128), float("nan"), dtype=torch.bfloat16, device=device)
        self.lse = torch.full((T, Hq), float("nan"), device=device)
        self.ws_bytes = msa_workspace_bytes(self.shape)
        if self.ws_bytes == 0:
            raise ValueError("shape rejected by msa_workspace_bytes")
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        msa_workspace_init(self.ws, self.ws_bytes)

    def replicate(self) -> "DeviceProblem":
        """A copy of every buffer at new device addresses (same bytes)."""
        import copy

        import torch

        dp = copy.copy(self)
        for name in ("q_idx", "idxk", "idxk_scales", "q", "kv", "block_table", "seq_lens",
                     "block_scores", "selected", "out", "lse"):
            t = getattr(self, name)
            setattr(dp, name, None if t is None else t.clone())
        dp.shape = type(self.shape).from_buffer_copy(self.shape)
        dp.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        msa_workspace_init(dp.ws, dp.ws_bytes)
        return dp

    def set_decode_ctas(self, n: int):
        import torch

        self.shape.decode_ctas = int(n)
        need = msa_workspace_bytes(self.shape)
        if need > self.ws_bytes:
            self.ws_bytes = need
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.device)
            msa_workspace_init(self.ws, need)

    # ---- the four entry points ----
    def index_score(self, stream=None):
        msa_index_score(self.shape, self.q_idx, self.idxk, self.idxk_scales, self.block_table,
                        self.seq_lens, self.block_scores, self.ws, self.ws_bytes, stream)

    def select(self, block_scores=None, stream=None):
        bs = self.block_scores if block_scores is None else block_scores
        msa_select_topk(self.shape, bs, self.seq_lens, self.selected, self.ws, self.ws_bytes,
                        stream)

    def sparse_decode(self, selected=None, stream=None):
        sel = self.selected if selected is None else selected
        msa_sparse_decode(self.shape, self.q, self.kv, self.block_table, self.seq_lens, sel,
                          self.out, self.lse, self.ws, self.ws_bytes, stream)

    def decode_step(self, keep_intermediates: bool = True, stream=None):
        msa_decode_step(self.shape, self.q_idx, self.idxk, self.idxk_scales, self.q, self.kv,
                        self.block_table, self.seq_lens,
                        self.block_scores if keep_intermediates else None,
                        self.selected if keep_intermediates else None,
                        self.out, self.lse, self.ws, self.ws_bytes, stream)

    def kv_update(self, update: dict, stream=None):
        """Write this step's new tokens (synth.make_update arrays) into the pools."""
        self.k_new = _dev(update["k_new"], self.device)
        self.v_new = _dev(update["v_new"], self.device)
        self.idxk_new = _dev(update["idxk_new"], self.device)
        msa_kv_update(self.shape, self.k_new, self.v_new, self.idxk_new, self.block_table,
                      self.seq_lens, self.kv, self.idxk, self.idxk_scales, self.ws, self.ws_bytes,
                      stream)

    def pools(self) -> dict:
        """The pools as numpy arrays (the byte layouts of the synthetic module)."""
        import torch

        torch.cuda.synchronize()

        def host(t, like):
            a = t.cpu().numpy()
            return a.view(np.uint16) if like.dtype == np.uint16 else a

        return {"kv_pool": host(self.kv, self.pb.kv_pool),
                "idxk_pool": host(self.idxk, self.pb.idxk_pool),
                "idxk_scales": None if self.idxk_scales is None else self.idxk_scales.cpu().numpy()}

    # ---- results as numpy ----
    def results(self) -> dict:
        import torch

        torch.cuda.synchronize()
        one = self.shape.num_index_heads == 1   # one index head: [T, maxB] and [T, k]
        return {
            "block_scores": (self.block_scores[:, 0] if one else self.block_scores).cpu().numpy(),
            "selected": (self.selected[:, 0] if one else self.selected).cpu().numpy(),
            "out": self.out.float().cpu().numpy().astype(np.float64),
            "lse": self.lse.cpu().numpy().astype(np.float64),
        }
