"""A seeded workload resident on the GPU: the paged pool populated through
``splash_kv_append``, plus the step inputs (the verify block's K/V and Q).

Used by the benchmark, the smoke check and the GPU tests. Unused page bytes
are poisoned (codes +-127, scales NaN / inf) so that any read of a slot the
method must not touch shows up in the output.
"""
from __future__ import annotations

import numpy as np
import torch

from . import splash_kv as sk
from . import workloads as wl

POISON_CODE = 127


def _stack_heads(pairs):
    ks, vs = zip(*pairs)
    return np.stack(ks, axis=1), np.stack(vs, axis=1)


class DeviceWorkload:
    def __init__(self, W: wl.Workload, seqs=None, populate: bool = True, device="cuda",
                 chunk_tokens: int = 16384):
        self.W = W
        s = W.spec
        self.device = device
        kp, vp, ks, vs = sk.alloc_pool(W.num_pages, s.num_kv_heads, s.head_dim, device)
        kp.fill_(POISON_CODE)
        vp.fill_(-POISON_CODE)
        ks.fill_(float("nan"))
        vs.fill_(float("inf"))
        self.pool = (kp, vp, ks, vs)
        self.table = torch.from_numpy(W.page_table).to(device)
        self.ctx = torch.from_numpy(W.context_lens).to(device)
        self.T = torch.from_numpy(W.block_lens).to(device)
        self.max_T = max(int(W.block_lens.max()) if W.num_seqs else 0, 1)
        bk, bv = W.block_kv()
        self.k_new = torch.from_numpy(bk).to(device)
        self.v_new = torch.from_numpy(bv).to(device)
        self.q = torch.from_numpy(W.q_bits().view(np.int16)).to(device).view(torch.bfloat16)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # sequences that share a prefix go through the shared-prefix entry point
        # (the prefix read once per row block of the stacked rows)
        self.shared_lens = (torch.from_numpy(W.shared_lens()).to(device) if W.prefix_len
                            else None)
        self.ws = sk.alloc_workspace(W.num_seqs, W.num_q_tokens, s.num_q_heads, s.num_kv_heads,
                                     s.head_dim, self.max_T, device=device,
                                     shared=self.shared_lens is not None)
        if populate:
            self.populate(seqs, chunk_tokens)

    # ---- cache population (setup, not part of a step) -------------------
    def _append(self, k, v, b, start):
        n = k.shape[0]
        if n == 0:
            return
        sk.splash_kv_append(torch.from_numpy(np.ascontiguousarray(k)).to(self.device),
                            torch.from_numpy(np.ascontiguousarray(v)).to(self.device),
                            *self.pool, self.table[b:b + 1],
                            torch.tensor([start], dtype=torch.int32, device=self.device),
                            torch.tensor([n], dtype=torch.int32, device=self.device),
                            device_status=self.status)

    def populate(self, seqs=None, chunk_tokens: int = 16384):
        """Append the cached context of ``seqs`` (all by default); a shared
        prefix is appended once, through the first sequence's page list."""
        W = self.W
        H = W.spec.num_kv_heads
        seqs = range(W.num_seqs) if seqs is None else list(seqs)
        if W.prefix_len:
            k, v = _stack_heads([W.prefix_kv(h) for h in range(H)])
            for c0 in range(0, k.shape[0], chunk_tokens):
                self._append(k[c0:c0 + chunk_tokens], v[c0:c0 + chunk_tokens], 0, c0)
        for b in seqs:
            k, v = _stack_heads([W.private_context_kv(b, h) for h in range(H)])
            for c0 in range(0, k.shape[0], chunk_tokens):
                self._append(k[c0:c0 + chunk_tokens], v[c0:c0 + chunk_tokens], b,
                             W.prefix_len + c0)
        torch.cuda.synchronize()
        if int(self.status.item()) != 0:
            raise RuntimeError(f"device status {int(self.status.item())} while populating")

    # ---- pool copies (to run steps on inputs that L2 cannot hold) --------
    def pool_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.pool[0]._base, self.pool[2], self.pool[3]))

    def add_pool_copies(self, n: int):
        """n identical pools in total; use_pool(i) selects copy i % n."""
        base = self.pool[0]._base
        self.pools = [self.pool]
        for _ in range(n - 1):
            codes = base.clone()
            self.pools.append((codes[:, :, 0], codes[:, :, 1], self.pool[2].clone(),
                               self.pool[3].clone()))

    def use_pool(self, i: int):
        pools = getattr(self, "pools", [self.pool])
        self.pool = pools[i % len(pools)]

    # ---- one step: append the verify block, attend ----------------------
    def append_block(self, stream=None):
        sk.splash_kv_append(self.k_new, self.v_new, *self.pool, self.table, self.ctx, self.T,
                            device_status=self.status, stream=stream)

    def attend(self, path=sk.PATH_AUTO, ctas=0, out=None, lse=None, stream=None, window=0,
               table=None, stack=True, events=None, shared_lens=None):
        """One verify-attention call. With a shared prefix (and no window) it
        goes through the shared-prefix entry point unless ``stack`` is False;
        ``shared_lens`` overrides the workload's own."""
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        sl = shared_lens if shared_lens is not None else self.shared_lens
        if not stack or window != 0:
            sl = None
        sk.splash_verify_attention(self.q, *self.pool, self.table if table is None else table,
                                   self.ctx, self.T, float(self.W.sm_scale), self.max_T, out, lse,
                                   self.ws, device_status=self.status, stream=stream, path=path,
                                   ctas_per_class=ctas, window=window, events=events,
                                   shared_lens=sl)
        return out, lse

    def step(self, stream=None):
        self.append_block(stream)
        return self.attend(stream=stream)
