"""Helpers for the GPU parity tests: move a generated case to the device and
run the library's calls on it. No attention arithmetic here."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_decode_gb300 as pkv
from paged_kv_decode_gb300.build import build_library

_built = False


def ensure_built():
    global _built
    if not _built:
        build_library()
        _built = True


def i32(a, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit pattern of a bf16 tensor (NaN payloads included)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class DecodeOnDevice:
    """One layer of a DecodeCase on the GPU, with a workspace."""

    def __init__(self, case, layer: int, device):
        ensure_built()
        self.case = case
        self.device = device
        self.q = case.q[layer].to(device)
        self.k_pages = case.k_pages[layer].to(device)
        self.v_pages = case.v_pages[layer].to(device)
        self.block_table = i32(case.block_table, device)
        self.seq_lens = i32(case.seq_lens, device)
        self.slot_mapping = i32(case.slot_mapping, device)
        self.k_new = None if case.k_new is None else case.k_new[layer].to(device)
        self.v_new = None if case.v_new is None else case.v_new[layer].to(device)
        self.out = torch.empty_like(self.q)
        g = case.geom
        nbytes = pkv.decode_workspace_bytes(case.batch, case.max_pages, case.num_pages, g.n_q_heads, g.n_kv_heads,
                                            g.head_dim)
        assert nbytes > 0
        self.ws = pkv.Workspace(nbytes, device)

    def step(self):
        if self.k_new is not None:
            pkv.append(self.k_new, self.v_new, self.slot_mapping, self.k_pages, self.v_pages, self.ws)
        pkv.decode_attn(self.q, self.k_pages, self.v_pages, self.block_table, self.seq_lens, self.out,
                        self.case.geom.scale, self.ws)
        return self.out

    def pools_cpu(self):
        return self.k_pages.cpu(), self.v_pages.cpu()
