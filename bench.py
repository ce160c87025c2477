#!/usr/bin/env python
"""Benchmark of the sink-aware varlen attention forward on GB300.

Default workload: the vision-tower window block at 16384 tokens (4 packed
sequences of 4096), 16 MHA heads, head dim 80, symmetric window 64, KEY0_BIAS
sinks -- the window-attention call whose H100 cost the MiMo sinks pull
request quotes.  One step = one call of the C-ABI entry point (all of the
forward runs inside its kernels).  Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

Other workloads (--workload): the 4096-token vision block, the 16384-token
GQA window, the sparse MLA decode (64 queries x 128 heads, top-2048 indices,
NULL_LOGIT) and the block-sparse DSA prefill (2 x 8192 tokens, top-16
blocks, NULL_LOGIT).

Timing: W untimed warm-up calls, then K calls bracketed by a barrier and
torch.cuda.synchronize(); each call is also bracketed by CUDA events on the
launching stream for its kernels' duration.  Several input sets rotate so that
the bytes touched between two calls of one set exceed the 129 MB L2.  SM
clocks and throttle reasons are sampled with nvidia-smi during the timed
region.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attention_head_sinks_gb300 import workloads as W  # noqa: E402

MODE_NAMES = {0: "NONE", 1: "KEY0_BIAS", 2: "NULL_LOGIT"}
L2_BYTES = 129 * 1024 * 1024
METRIC = "attn fwd us/call (achieved HBM GB/s as % of GB300 roofline)"
# The pages' cost of the same window call on H100 (FA varlen + post-hoc key-0
# sink correction, 16 heads, head dim 80, window 64).
PAGES_H100_US = {"vision_window_16384tok": 289.0, "vision_window_4096tok": 248.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def _torch_bits(a):
    return W.to_torch(a)


def _obufs(runner):
    """Output arrays the oracle keeps between the sampled calls of one
    runner, so that a sampled call does not allocate and fill full-size
    outputs (the arithmetic is the oracle's, unchanged)."""
    if not hasattr(runner, "_oracle_bufs"):
        runner._oracle_bufs = {}
    return runner._oracle_bufs


# ----------------------------------------------------------------------------
# workloads: inputs, algorithmic bytes / flops, the call, the oracle sample
# ----------------------------------------------------------------------------
class WindowRunner:
    """sa_varlen_window_fwd on a packed window workload."""
    bound = "hbm"
    # the persistent ring kernel serves every bench window workload (the
    # one-tile kernel in window_fwd.cu is the fallback for other shapes)
    source = "attention_head_sinks_gb300/csrc/window_ring_fwd.cu"


    oracle_kind = "fp64 C oracle with OpenMP"
    @staticmethod
    def oracle_cores():
        from oracle import sa_oracle
        return sa_oracle.num_threads()

    def __init__(self, name):
        self.name = name
        if name == "vision_window_16384tok":
            self.c = W.vision_window(16384, W.SINK_KEY0_BIAS)
        elif name == "vision_window_4096tok":
            self.c = W.vision_window(4096, W.SINK_KEY0_BIAS)
        elif name == "tiny_window_128tok":
            # launch-bound parity case: its inputs stay L2-resident
            self.bound = "launch"
            self.c = W.tiny_window(W.SINK_KEY0_BIAS)
        else:
            self.c = W.gqa_window(W.SINK_KEY0_BIAS)
        self.mode = self.c.mode

    def counts(self):
        """Bytes: q, o once; k, v once per KV head; LSE.  Flops: 4 * D per live
        (row, key, head)."""
        c = self.c
        T, hq, d = c.q.shape
        hkv = c.k.shape[1]
        nbytes = 2 * T * hq * d * 2 + 2 * T * hkv * d * 2 + hq * T * 4
        cu = c.cu_seqlens.astype(np.int64)
        live = 0
        for b in range(len(cu) - 1):
            n = int(cu[b + 1] - cu[b])
            i = np.arange(n)
            live += int((np.minimum(n - 1, i + c.window_right)
                         - np.maximum(0, i - c.window_left) + 1).sum())
        return nbytes, 4 * d * live * hq

    def config(self):
        c = self.c
        T, hq, d = c.q.shape
        return {"workload": self.name, "tokens": int(T),
                "seqs": int(len(c.cu_seqlens) - 1), "q_heads": int(hq),
                "kv_heads": int(c.k.shape[1]), "head_dim": int(d),
                "window": int(c.window_left), "sink_mode": MODE_NAMES[self.mode]}

    def setup(self, nsets):
        import torch
        c = self.c
        dev = torch.device("cuda")
        self.sets = []
        for _ in range(nsets):
            q, k, v = (_torch_bits(x).to(dev) for x in (c.q, c.k, c.v))
            out = torch.empty_like(q)
            lse = torch.empty((c.q.shape[1], c.q.shape[0]), dtype=torch.float32,
                              device=dev)
            self.sets.append((q, k, v, out, lse))
        self.cu = torch.from_numpy(c.cu_seqlens).to(dev)
        self.sinks = torch.from_numpy(c.sinks).to(dev)

    def touched_bytes(self):
        return self.counts()[0]

    def launches_per_call(self):
        return 1

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        q, k, v, out, lse = self.sets[i % len(self.sets)]
        c = self.c
        sa.sa_varlen_window_fwd(q, k, v, self.cu, c.window_left, c.window_right,
                                self.sinks, self.mode if mode is None else mode,
                                c.scale, out=out, lse=lse)

    def host_io(self, slot=0):
        import torch
        c = self.c
        host_in = [_torch_bits(x) for x in (c.q, c.k, c.v)] + \
            [torch.from_numpy(c.cu_seqlens), torch.from_numpy(c.sinks)]
        out, lse = self.sets[slot][3], self.sets[slot][4]

        def run(dev_in):
            import attention_head_sinks_gb300 as sa
            sa.sa_varlen_window_fwd(dev_in[0], dev_in[1], dev_in[2], dev_in[3],
                                    c.window_left, c.window_right, dev_in[4],
                                    self.mode, c.scale, out=out, lse=lse)
        return host_in, [out, lse], run

    def oracle_rows(self):
        return self.c.q.shape[0]

    def oracle(self, rows):
        from oracle import sa_oracle
        c = self.c
        sa_oracle.window_fwd(c.q, c.k, c.v, c.cu_seqlens, c.window_left,
                             c.window_right, c.sinks, self.mode, c.scale, rows=rows, bufs=_obufs(self))


class IndexRunner:
    """sa_sparse_index_fwd on the sparse MLA decode workload."""
    bound = "hbm"
    source = "attention_head_sinks_gb300/csrc/sparse_index_fwd.cu"


    oracle_kind = "fp64 C oracle with OpenMP"
    @staticmethod
    def oracle_cores():
        from oracle import sa_oracle
        return sa_oracle.num_threads()

    def __init__(self, name):
        self.name = name
        self.c = W.mla_sparse_decode(W.SINK_NULL_LOGIT)
        self.mode = self.c.mode

    def counts(self):
        """Bytes: q and o once, each listed (valid) latent row once per query,
        the index list and the LSE.  Flops: (2 dqk + 2 dv) per (query, head,
        valid key)."""
        c = self.c
        nq, hq, dqk = c.q.shape
        valid = int(((c.indices >= 0) & (c.indices < c.num_kv)).sum())
        nbytes = (nq * hq * dqk * 2 + nq * hq * c.dv * 2 + valid * dqk * 2
                  + c.indices.nbytes + hq * nq * 4)
        return nbytes, valid * hq * (2 * dqk + 2 * c.dv)

    def config(self):
        c = self.c
        return {"workload": self.name, "queries": c.num_queries,
                "q_heads": c.num_q_heads, "dqk": c.dqk, "dv": c.dv,
                "kv_rows": c.num_kv, "topk": c.topk,
                "valid_per_query": list(W.MLA_VALID_COUNTS),
                "sink_mode": MODE_NAMES[self.mode]}

    def setup(self, nsets):
        import torch
        import attention_head_sinks_gb300 as sa
        c = self.c
        dev = torch.device("cuda")
        self.sets = []
        for _ in range(nsets):
            q, kv = _torch_bits(c.q).to(dev), _torch_bits(c.kv).to(dev)
            idx = torch.from_numpy(c.indices).to(dev)
            out = torch.empty((c.num_queries, c.num_q_heads, c.dv),
                              dtype=torch.bfloat16, device=dev)
            lse = torch.empty((c.num_q_heads, c.num_queries), dtype=torch.float32,
                              device=dev)
            self.sets.append((q, kv, idx, out, lse))
        self.sinks = torch.from_numpy(c.sinks).to(dev)
        self.ws = torch.empty(max(1, sa.sa_sparse_index_workspace_size(
            c.num_queries, c.num_q_heads, c.dv, c.topk)), dtype=torch.uint8, device=dev)

    def touched_bytes(self):
        return self.counts()[0]

    def launches_per_call(self):
        # plan, then the persistent attend kernel (split-KV merge included)
        return 2

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        q, kv, idx, out, lse = self.sets[i % len(self.sets)]
        c = self.c
        sa.sa_sparse_index_fwd(q, kv, idx, c.dv, self.sinks,
                               self.mode if mode is None else mode, c.scale,
                               out=out, lse=lse, workspace=self.ws)

    def host_io(self, slot=0):
        import torch
        c = self.c
        host_in = [_torch_bits(c.q), _torch_bits(c.kv), torch.from_numpy(c.indices),
                   torch.from_numpy(c.sinks)]
        out, lse = self.sets[slot][3], self.sets[slot][4]
        # a second slot runs concurrently: its own split-KV workspace
        ws = self.ws if slot == 0 else torch.empty_like(self.ws)

        def run(dev_in):
            import attention_head_sinks_gb300 as sa
            sa.sa_sparse_index_fwd(dev_in[0], dev_in[1], dev_in[2], c.dv, dev_in[3],
                                   self.mode, c.scale, out=out, lse=lse, workspace=ws)
        return host_in, [out, lse], run

    def oracle_rows(self):
        return self.c.num_queries

    def oracle(self, rows):
        from oracle import sa_oracle
        c = self.c
        sa_oracle.sparse_index_fwd(c.q, c.kv, c.indices, c.dv, c.sinks, self.mode,
                                   c.scale, rows=rows, bufs=_obufs(self))


class IndexFp8Runner(IndexRunner):
    """sa_sparse_index_fwd_fp8 on the sparse MLA decode workload over an e4m3
    latent cache with one fp32 scale per row."""
    oracle_kind = "fp64 numpy oracle (one query per step)"

    @staticmethod
    def oracle_cores():
        try:
            import threadpoolctl
            n = [i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()
                 if i.get("user_api") == "blas"]
            if n:
                return int(max(n))
        except ImportError:
            pass
        return os.cpu_count() or 1

    def __init__(self, name):
        self.name = name
        self.c = W.mla_sparse_decode_fp8(W.SINK_NULL_LOGIT)
        self.mode = self.c.mode

    def counts(self):
        """Bytes: q and o once, each listed (valid) e4m3 latent row and its
        fp32 scale once per query, the index list and the LSE.  Flops as the
        bf16 cache."""
        c = self.c
        nq, hq, dqk = c.q.shape
        valid = int(((c.indices >= 0) & (c.indices < c.num_kv)).sum())
        nbytes = (nq * hq * dqk * 2 + nq * hq * c.dv * 2 + valid * (dqk + 4)
                  + c.indices.nbytes + hq * nq * 4)
        return nbytes, valid * hq * (2 * dqk + 2 * c.dv)

    def config(self):
        cfg = super().config()
        cfg["kv_cache"] = "e4m3 codes + fp32 scale per row"
        return cfg

    def setup(self, nsets):
        import torch
        import attention_head_sinks_gb300 as sa
        c = self.c
        dev = torch.device("cuda")
        self.sets = []
        for _ in range(nsets):
            q = _torch_bits(c.q).to(dev)
            kv = torch.from_numpy(c.kv).to(dev)
            ks = torch.from_numpy(c.kv_scale).to(dev)
            idx = torch.from_numpy(c.indices).to(dev)
            out = torch.empty((c.num_queries, c.num_q_heads, c.dv),
                              dtype=torch.bfloat16, device=dev)
            lse = torch.empty((c.num_q_heads, c.num_queries), dtype=torch.float32,
                              device=dev)
            self.sets.append((q, kv, ks, idx, out, lse))
        self.sinks = torch.from_numpy(c.sinks).to(dev)
        self.ws = torch.empty(max(1, sa.sa_sparse_index_workspace_size(
            c.num_queries, c.num_q_heads, c.dv, c.topk)), dtype=torch.uint8, device=dev)

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        q, kv, ks, idx, out, lse = self.sets[i % len(self.sets)]
        c = self.c
        sa.sa_sparse_index_fwd_fp8(q, kv, ks, idx, c.dv, self.sinks,
                                   self.mode if mode is None else mode, c.scale,
                                   out=out, lse=lse, workspace=self.ws)

    def host_io(self, slot=0):
        import torch
        c = self.c
        host_in = [_torch_bits(c.q), torch.from_numpy(c.kv), torch.from_numpy(c.kv_scale),
                   torch.from_numpy(c.indices), torch.from_numpy(c.sinks)]
        out, lse = self.sets[slot][4], self.sets[slot][5]
        # a second slot runs concurrently: its own split-KV workspace
        ws = self.ws if slot == 0 else torch.empty_like(self.ws)

        def run(dev_in):
            import attention_head_sinks_gb300 as sa
            sa.sa_sparse_index_fwd_fp8(dev_in[0], dev_in[1], dev_in[2], dev_in[3], c.dv,
                                       dev_in[4], self.mode, c.scale, out=out, lse=lse,
                                       workspace=ws)
        return host_in, [out, lse], run

    def oracle(self, rows):
        from oracle import sa_oracle
        c = self.c
        sa_oracle.sparse_index_fwd_fp8(c.q, c.kv, c.kv_scale, c.indices, c.dv, c.sinks,
                                       self.mode, c.scale, rows=rows, bufs=_obufs(self))


class BlockRunner:
    """sa_block_sparse_fwd on the DSA-style block-sparse prefill."""
    bound = "tensor"
    source = "attention_head_sinks_gb300/csrc/block_sparse_fwd.cu"


    oracle_kind = "fp64 C oracle with OpenMP"
    @staticmethod
    def oracle_cores():
        from oracle import sa_oracle
        return sa_oracle.num_threads()

    def __init__(self, name):
        self.name = name
        # dsa_block_prefill_key0: the same batch with KEY0_BIAS sinks on the
        # first key of each document
        mode = W.SINK_KEY0_BIAS if name.endswith("_key0") else W.SINK_NULL_LOGIT
        self.c = W.dsa_block_prefill(mode)
        self.mode = self.c.mode

    def counts(self):
        """Bytes: q, o once; k, v once per KV head; table; LSE.  Flops counted
        over the selected blocks: 4 * D * 64 per (token, head, selected
        block)."""
        c = self.c
        T, hq, d = c.q.shape
        hkv = c.k.shape[1]
        nbytes = 2 * T * hq * d * 2 + 2 * T * hkv * d * 2 + c.block_table.nbytes + hq * T * 4
        nsel = int(((c.block_table >= 0) & (c.block_table < c.seq_len // c.block_size)).sum())
        return nbytes, nsel * c.block_size * hq * 4 * d

    def config(self):
        c = self.c
        return {"workload": self.name, "batch": c.batch, "seq_len": c.seq_len,
                "q_heads": c.num_q_heads, "kv_heads": c.num_kv_heads,
                "head_dim": c.head_dim, "block_size": c.block_size,
                "topk_blocks": c.topk_blocks, "docs_per_row": 3,
                "sink_mode": MODE_NAMES[self.mode],
                "flops_basis": "selected blocks"}

    def setup(self, nsets):
        import torch
        c = self.c
        dev = torch.device("cuda")
        self.sets = []
        for _ in range(nsets):
            q, k, v = (_torch_bits(x).to(dev) for x in (c.q, c.k, c.v))
            out = torch.empty_like(q)
            lse = torch.empty((c.num_q_heads, c.total_tokens), dtype=torch.float32,
                              device=dev)
            self.sets.append((q, k, v, out, lse))
        self.table = torch.from_numpy(c.block_table).to(dev)
        self.cu = torch.from_numpy(c.cu_docs).to(dev)
        self.sinks = torch.from_numpy(c.sinks).to(dev)

    def touched_bytes(self):
        return self.counts()[0]

    def launches_per_call(self):
        return 1

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        q, k, v, out, lse = self.sets[i % len(self.sets)]
        c = self.c
        sa.sa_block_sparse_fwd(q, k, v, c.batch, c.seq_len, self.table, c.block_size,
                               self.cu, self.sinks, self.mode if mode is None else mode,
                               c.scale, out=out, lse=lse)

    def host_io(self, slot=0):
        import torch
        c = self.c
        host_in = [_torch_bits(x) for x in (c.q, c.k, c.v)] + \
            [torch.from_numpy(c.block_table), torch.from_numpy(c.cu_docs),
             torch.from_numpy(c.sinks)]
        out, lse = self.sets[slot][3], self.sets[slot][4]

        def run(dev_in):
            import attention_head_sinks_gb300 as sa
            sa.sa_block_sparse_fwd(dev_in[0], dev_in[1], dev_in[2], c.batch, c.seq_len,
                                   dev_in[3], c.block_size, dev_in[4], dev_in[5],
                                   self.mode, c.scale, out=out, lse=lse)
        return host_in, [out, lse], run

    def oracle_rows(self):
        return self.c.total_tokens

    def oracle(self, rows):
        from oracle import sa_oracle
        c = self.c
        sa_oracle.block_sparse_fwd(c.q, c.k, c.v, c.batch, c.seq_len, c.block_table,
                                   c.block_size, c.cu_docs, c.sinks, self.mode,
                                   c.scale, rows=rows, bufs=_obufs(self))


class MergeRunner:
    """sa_merge_attn_states on two window-block-shaped partials."""
    bound = "hbm"

    source = "attention_head_sinks_gb300/csrc/merge_states.cu"

    oracle_kind = "fp64 NumPy oracle"
    @staticmethod
    def oracle_cores():
        return 1  # the merge oracle is single-threaded NumPy

    def __init__(self, name):
        self.name = name
        self.c = W.merge_window_partials(W.SINK_NULL_LOGIT)
        self.mode = self.c.mode

    def counts(self):
        """Bytes: both partial outputs and LSEs read once, the merged output
        and LSE written once.  Flops: 3 per output element (two scaled
        terms and their sum)."""
        c = self.c
        T, h, d = c.out_a.shape
        return 3 * T * h * d * 2 + 3 * h * T * 4, 3 * T * h * d

    def config(self):
        T, h, d = self.c.out_a.shape
        return {"workload": self.name, "tokens": int(T), "heads": int(h), "head_dim": int(d),
                "sink_mode": MODE_NAMES[self.mode]}

    def setup(self, nsets):
        import torch
        c = self.c
        dev = torch.device("cuda")
        self.sets = []
        for _ in range(nsets):
            oa, ob = _torch_bits(c.out_a).to(dev), _torch_bits(c.out_b).to(dev)
            la, lb = torch.from_numpy(c.lse_a).to(dev), torch.from_numpy(c.lse_b).to(dev)
            out = torch.empty_like(oa)
            lse = torch.empty_like(la)
            self.sets.append((oa, la, ob, lb, out, lse))
        self.sinks = torch.from_numpy(c.sinks).to(dev)

    def touched_bytes(self):
        return self.counts()[0]

    def launches_per_call(self):
        return 1

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        oa, la, ob, lb, out, lse = self.sets[i % len(self.sets)]
        sa.sa_merge_attn_states(oa, la, ob, lb, self.sinks,
                                self.mode if mode is None else mode, out=out, lse=lse)

    def host_io(self, slot=0):
        import torch
        c = self.c
        host_in = [_torch_bits(c.out_a), torch.from_numpy(c.lse_a), _torch_bits(c.out_b),
                   torch.from_numpy(c.lse_b), torch.from_numpy(c.sinks)]
        out, lse = self.sets[slot][4], self.sets[slot][5]

        def run(dev_in):
            import attention_head_sinks_gb300 as sa
            sa.sa_merge_attn_states(dev_in[0], dev_in[1], dev_in[2], dev_in[3], dev_in[4],
                                    self.mode, out=out, lse=lse)
        return host_in, [out, lse], run

    def oracle_rows(self):
        return self.c.out_a.shape[0]

    def oracle(self, rows):
        from oracle import sa_oracle
        c = self.c
        b, e = rows
        sa_oracle.merge_states(c.out_a[b:e], c.lse_a[:, b:e], c.out_b[b:e], c.lse_b[:, b:e],
                               c.sinks, self.mode)


class SelectRunner:
    """sa_block_select on the indexer inputs of the DSA prefill batch."""
    bound = "tensor"
    source = "attention_head_sinks_gb300/csrc/block_select.cu"
    oracle_kind = "fp64 numpy oracle (one token per step)"

    @staticmethod
    def oracle_cores():
        return IndexFp8Runner.oracle_cores()

    def __init__(self, name):
        self.name = name
        self.c = W.dsa_block_select()
        self.mode = W.SINK_NONE

    def counts(self):
        """Bytes: index q, index k and the table once.  Flops: 2 * Di per
        (token, index head, key of a block before the token's own)."""
        c = self.c
        T, hi, di = c.index_q.shape
        pos = np.arange(T) % c.seq_len
        keys = int(((pos // c.block_size) * c.block_size).sum())
        nbytes = c.index_q.nbytes + c.index_k.nbytes + hi * T * c.topk * 4
        return nbytes, keys * hi * 2 * di

    def config(self):
        c = self.c
        return {"workload": self.name, "batch": c.batch, "seq_len": c.seq_len,
                "index_heads": c.num_index_heads, "index_dim": c.index_dim,
                "block_size": c.block_size, "topk_blocks": c.topk,
                "flops_basis": "keys of the blocks each token ranks"}

    def setup(self, nsets):
        import torch
        c = self.c
        dev = torch.device("cuda")
        T = c.batch * c.seq_len
        self.sets = []
        for _ in range(nsets):
            qi, ki = _torch_bits(c.index_q).to(dev), _torch_bits(c.index_k).to(dev)
            tab = torch.empty((c.num_index_heads, T, c.topk), dtype=torch.int32, device=dev)
            self.sets.append((qi, ki, tab))

    def touched_bytes(self):
        return self.counts()[0]

    def launches_per_call(self):
        return 1

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        qi, ki, tab = self.sets[i % len(self.sets)]
        c = self.c
        sa.sa_block_select(qi, ki, c.batch, c.seq_len, c.block_size, c.topk, block_table=tab)

    def host_io(self, slot=0):
        c = self.c
        host_in = [_torch_bits(c.index_q), _torch_bits(c.index_k)]
        tab = self.sets[slot][2]

        def run(dev_in):
            import attention_head_sinks_gb300 as sa
            sa.sa_block_select(dev_in[0], dev_in[1], c.batch, c.seq_len, c.block_size, c.topk,
                               block_table=tab)
        return host_in, [tab], run

    def oracle_rows(self):
        return self.c.batch * self.c.seq_len

    def oracle(self, rows):
        from oracle import sa_oracle
        c = self.c
        sa_oracle.block_select(c.index_q, c.index_k, c.batch, c.seq_len, c.block_size, c.topk,
                               rows=rows, bufs=_obufs(self))


class SelectedBlockRunner(BlockRunner):
    """The DSA prefill step with its selection made on the device:
    sa_block_select (4 index heads, one per KV head) then
    sa_block_sparse_fwd_index_heads with those tables."""
    oracle_kind = "fp64 numpy selection + fp64 C attention oracle with OpenMP"

    def __init__(self, name):
        super().__init__(name)
        self.sc = W.dsa_block_select()

    def counts(self):
        """Bytes: the attention's (q, o, k, v, LSE) plus the indexer inputs
        and the table.  Flops: the selection's plus the attention's over the
        selected blocks, which are those of the tables the selection writes
        (their count is fixed by the shape: every token selects
        min(own block + 1, topk) blocks)."""
        c, sc = self.c, self.sc
        T, hq, d = c.q.shape
        hkv = c.k.shape[1]
        pos = np.arange(T) % c.seq_len
        nsel = np.minimum(pos // c.block_size + 1, sc.topk)
        hi = sc.num_index_heads
        att_flops = int(nsel.sum()) * c.block_size * hq * 4 * d
        keys = int(((pos // sc.block_size) * sc.block_size).sum())
        sel_flops = keys * hi * 2 * sc.index_dim
        nbytes = (2 * T * hq * d * 2 + 2 * T * hkv * d * 2 + hq * T * 4 + sc.index_q.nbytes
                  + sc.index_k.nbytes + 2 * hi * T * sc.topk * 4)
        return nbytes, att_flops + sel_flops

    def config(self):
        cfg = super().config()
        cfg.update({"index_heads": self.sc.num_index_heads, "index_dim": self.sc.index_dim,
                    "selection": "on device (sa_block_select)",
                    "flops_basis": "selected blocks + selection scores"})
        return cfg

    def setup(self, nsets):
        import torch
        super().setup(nsets)
        sc = self.sc
        dev = torch.device("cuda")
        T = sc.batch * sc.seq_len
        self.qi, self.ki = _torch_bits(sc.index_q).to(dev), _torch_bits(sc.index_k).to(dev)
        self.tabs = torch.empty((sc.num_index_heads, T, sc.topk), dtype=torch.int32,
                                device=dev)

    def launches_per_call(self):
        return 2

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        q, k, v, out, lse = self.sets[i % len(self.sets)]
        c, sc = self.c, self.sc
        sa.sa_block_select(self.qi, self.ki, sc.batch, sc.seq_len, sc.block_size, sc.topk,
                           block_table=self.tabs)
        sa.sa_block_sparse_fwd_index_heads(q, k, v, c.batch, c.seq_len, self.tabs,
                                           c.block_size, self.cu, self.sinks,
                                           self.mode if mode is None else mode, c.scale,
                                           out=out, lse=lse)

    def host_io(self, slot=0):
        import torch
        c, sc = self.c, self.sc
        host_in = [_torch_bits(x) for x in (c.q, c.k, c.v)] + \
            [_torch_bits(sc.index_q), _torch_bits(sc.index_k), torch.from_numpy(c.cu_docs),
             torch.from_numpy(c.sinks)]
        out, lse = self.sets[slot][3], self.sets[slot][4]
        tabs = self.tabs if slot == 0 else torch.empty_like(self.tabs)

        def run(dev_in):
            import attention_head_sinks_gb300 as sa
            sa.sa_block_select(dev_in[3], dev_in[4], sc.batch, sc.seq_len, sc.block_size,
                               sc.topk, block_table=tabs)
            sa.sa_block_sparse_fwd_index_heads(dev_in[0], dev_in[1], dev_in[2], c.batch,
                                               c.seq_len, tabs, c.block_size, dev_in[5],
                                               dev_in[6], self.mode, c.scale, out=out,
                                               lse=lse)
        return host_in, [out, lse], run

    def oracle(self, rows):
        from oracle import sa_oracle
        c, sc = self.c, self.sc
        tabs, _ = sa_oracle.block_select(sc.index_q, sc.index_k, sc.batch, sc.seq_len,
                                         sc.block_size, sc.topk, rows=rows, bufs=_obufs(self))
        sa_oracle.block_sparse_fwd_index_heads(c.q, c.k, c.v, c.batch, c.seq_len, tabs,
                                               c.block_size, c.cu_docs, c.sinks, self.mode,
                                               c.scale, rows=rows, bufs=_obufs(self))


RUNNERS = {
    "tiny_window_128tok": WindowRunner,
    "vision_window_16384tok": WindowRunner,
    "vision_window_4096tok": WindowRunner,
    "gqa_window_16384tok": WindowRunner,
    "mla_sparse_decode": IndexRunner,
    "mla_sparse_decode_fp8": IndexFp8Runner,
    "dsa_block_prefill": BlockRunner,
    "dsa_block_prefill_key0": BlockRunner,
    "merge_window_16384tok": MergeRunner,
    "dsa_block_select": SelectRunner,
    "dsa_block_prefill_selected": SelectedBlockRunner,
}


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples every 100 ms while it runs: SM clock, power, GPU
    utilisation and the throttle reasons.  A sample counts as under load when
    the GPU reports at least 50 % utilisation; the SM clock median is taken
    over those samples."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
               "sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, load_sm, power, reasons = [], [], [], [], set()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                clk, cmax = float(f[1]), float(f[2])
            except ValueError:
                continue
            sm.append(clk)
            smax.append(cmax)
            try:
                util = float(f[4])
            except ValueError:
                util = 0.0
            if util >= 50.0:
                load_sm.append(clk)
                try:
                    power.append(float(f[3]))
                except ValueError:
                    pass
                # throttle reasons count while the GPU works
                for name, val in zip(self.REASONS, f[6:10]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(load_sm) if load_sm else None,
                "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(load_sm),
                "sm_mhz_min_under_load": min(load_sm) if load_sm else None,
                "power_w_median_under_load": statistics.median(power) if power else None}


def gpu_uuid():
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(
            torch.cuda.current_device()).uuid)
    except Exception:
        return str(torch.cuda.current_device())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_sources(path):
    """The kernel file and every local header it includes (transitively,
    ``#include "..."``), the file first and the headers in path order."""
    import re
    seen, todo, heads = set(), [os.path.join(ROOT, path)], []
    while todo:
        f = os.path.normpath(todo.pop())
        if f in seen or not os.path.exists(f):
            continue
        seen.add(f)
        if f != os.path.normpath(os.path.join(ROOT, path)):
            heads.append(f)
        for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', open(f).read(), re.M):
            todo.append(os.path.join(os.path.dirname(f), inc))
    return [os.path.normpath(os.path.join(ROOT, path))] + sorted(heads)


def kernel_source_hash(path):
    """Hash of the kernel file together with the local headers it includes,
    so that a change in a shared header also invalidates recorded traffic."""
    h = hashlib.sha256()
    for f in kernel_sources(path):
        h.update(os.path.relpath(f, ROOT).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def recorded_traffic(workload, src_hash):
    """DRAM bytes per launch of the dominant kernel from an ncu capture
    summarised in profiles/dram_traffic.txt, valid only for the same kernel
    source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == workload \
                and f[1] == src_hash:
            return int(float(f[2]))
    return None


def max_over_ranks(value, dist, device):
    """The slowest rank's value (the whole job's step time); ``value`` itself
    without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value_us(step_ms, world):
    """us per call over the whole job: every rank runs one call per step, so
    the job completes ``world`` calls per slowest-rank step."""
    return step_ms * 1000.0 / world


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------
def _oracle_time(runner, rows):
    t0 = time.perf_counter()
    runner.oracle(rows)
    return time.perf_counter() - t0


def sample_spans(total, nrows, nspans=8):
    """``nspans`` equal spans spread evenly over [0, total), ``nrows`` rows in
    all (so the sample sees every part of the workload)."""
    per = max(1, nrows // nspans)
    step = max(per, total // nspans)
    return [(s, min(total, s + per)) for s in range(0, total, step)][:nspans]


def cpu_baseline(runner, budget_s=10.0):
    from oracle import sa_oracle
    total = runner.oracle_rows()
    probe = sample_spans(total, max(8, total // 64))
    dt = sum(_oracle_time(runner, r) for r in probe)
    nprobe = sum(e - s for s, e in probe)
    want = int(nprobe * budget_s / max(dt, 1e-6))
    nrows = int(min(total, max(nprobe, want)))
    spans = sample_spans(total, nrows)
    dt = sum(_oracle_time(runner, r) for r in spans)
    n = sum(e - s for s, e in spans)
    us = dt * 1e6 * total / n
    return {"value": round(us, 1), "unit": "us/call", "cores": runner.oracle_cores(),
            "kind": "oracle",
            "sample": "%d of %d query rows in %d evenly spread spans (all heads), %s; "
                      "scaled to one call" % (n, total, len(spans), runner.oracle_kind)}


def arm_config(runner, world):
    """The ``config`` object of a bench line (both arms): the workload's own
    keys, the job layout and the L2 hygiene of the timed region."""
    cfg = runner.config()
    nsets = input_sets(runner)
    if getattr(runner, "bound", "") == "launch":
        l2 = ("%d rotating input sets (%.1f MB touched), L2-resident: a launch-bound "
              "parity case" % (nsets, nsets * runner.touched_bytes() / 1e6))
    else:
        l2 = ("%d rotating input sets (%.0f MB touched) > 129 MB L2" %
              (nsets, nsets * runner.touched_bytes() / 1e6))
    cfg.update({"global_batch": world, "parallelism": "replicas x%d" % world, "l2": l2})
    return cfg


def input_sets(runner):
    """Input sets rotated between calls so that every call touches more than
    L2 since the last use of its set (at most 64 sets)."""
    return int(min(64, max(2, -(-3 * L2_BYTES // runner.touched_bytes()))))


def run_reference(args, rank):
    if rank != 0:
        return
    runner = RUNNERS[args.workload](args.workload)
    total = runner.oracle_rows()
    per = max(1, total // 128)           # each step: 1/128 of the call's rows
    nspan = max(1, total // per)
    starts = [((i % nspan) * per) for i in range(args.steps + args.warmup)]
    for s in starts[:args.warmup]:
        _oracle_time(runner, (s, min(total, s + per)))
    t0 = time.perf_counter()
    for s in starts[args.warmup:]:
        _oracle_time(runner, (s, min(total, s + per)))
    dt = time.perf_counter() - t0
    us_call = dt * 1e6 / max(args.steps, 1) * (total / per)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us_call, 1),
        "unit": "us/call", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": arm_config(runner, args.gpus),
        "cpu_baseline": {"value": round(us_call, 1), "unit": "us/call",
                         "cores": runner.oracle_cores(), "kind": "oracle",
                         "sample": "each step %d of %d query rows (all heads), walking "
                                   "the call in order; value scaled to one call"
                                   % (per, total)},
        "e2e": {"value": round(us_call, 1), "unit": "us/call",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the default run also measures every other configuration of the workload set
# (and the two composite steps), each on its own inputs; windows and decodes
# with these many calls, the prefills with fewer
EXTRA_WORKLOADS = [
    ("tiny_window_128tok", 2000),
    ("vision_window_4096tok", 2000),
    ("gqa_window_16384tok", 1000),
    ("mla_sparse_decode", 1000),
    ("mla_sparse_decode_fp8", 1000),
    ("dsa_block_prefill", 100),
    ("dsa_block_prefill_selected", 100),
]
SUSTAINED_S = 1.5


class Bench:
    """Measurement of one workload on this rank (CUDA events on the launching
    stream, max over ranks)."""

    def __init__(self, runner, dist, world):
        import torch
        self.torch = torch
        self.r = runner
        self.dist = dist
        self.world = world
        self.nbytes, self.flops = runner.counts()
        self.nsets = input_sets(runner)
        runner.setup(self.nsets)

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def warm(self, n):
        for i in range(n):
            self.r.call(i)
        self.barrier()

    def timed(self, mode, steps):
        """The contract's timed region: ``steps`` calls through the public
        API, bracketed by barrier + synchronize, CUDA events on the launching
        stream at both ends; nothing else is enqueued in between.  The calls
        are queued behind a device-side sleep recorded before the first event,
        so that the host's enqueue time of the first calls never shows as idle
        device time inside the region (it is measured by the end-to-end leg).
        Returns the slowest rank's milliseconds."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.barrier()
        sleep = getattr(torch.cuda, "_sleep", None)
        if sleep is not None:  # about 30 us of host time per queued call
            sleep(int(2.0e9 * (0.002 + min(steps, 2000) * 30e-6)))
        gc_was = gc.isenabled()
        gc.disable()  # a collection pause longer than the sleep would idle the device
        try:
            e0.record()
            for i in range(steps):
                self.r.call(i, mode)
            e1.record()
        finally:
            if gc_was:
                gc.enable()
        self.barrier()
        return max_over_ranks(e0.elapsed_time(e1), self.dist, "cuda")

    def device_times(self, mode, steps):
        """Device time of each call (CUDA events around it on the launching
        stream), with the calls queued behind a device-side sleep so that the
        host's enqueue time never appears as idle time between the events."""
        torch = self.torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        self.barrier()
        sleep = getattr(torch.cuda, "_sleep", None)
        if sleep is not None:  # about 60 us of host time per queued call
            sleep(int(2.0e9 * (0.005 + steps * 60e-6)))
        gc_was = gc.isenabled()
        gc.disable()
        try:
            for i in range(steps):
                starts[i].record()
                self.r.call(i, mode)
                ends[i].record()
        finally:
            if gc_was:
                gc.enable()
        self.barrier()
        return [s_.elapsed_time(e_) * 1000.0 for s_, e_ in zip(starts, ends)]

    def sink_cost(self, steps):
        """Timed regions of back-to-back calls in the workload's mode and with
        sinks disabled, in alternating rounds so that a drift in clocks or in
        the machine's other load falls on both alike (the ratio of the two
        modes' median rounds); and the medians of isolated launches of both
        modes, alternating in the same way."""
        rounds = 4
        per_round = max(steps // rounds, 10)
        t_modes, t_nones = [], []
        for _ in range(rounds):
            t_modes.append(self.timed(self.r.mode, per_round))
            t_nones.append(self.timed(W.SINK_NONE, per_round))
        # medians over the rounds: one round disturbed by the host (a pause
        # longer than the device sleep ahead of it) does not count
        t_mode, t_none = statistics.median(t_modes), statistics.median(t_nones)
        ndev = max(min(steps, 500), 10)
        chunk = min(ndev, 50)
        per, per_none = [], []
        for _ in range((ndev + chunk - 1) // chunk):
            per += self.device_times(self.r.mode, chunk)
            per_none += self.device_times(W.SINK_NONE, chunk)
        kern, kern_none = statistics.median(per), statistics.median(per_none)
        return {"sink_cost": round(t_mode / t_none - 1.0, 4),
                "sink_cost_isolated": round(kern / kern_none - 1.0, 4),
                "launch_us_isolated": round(kern, 3),
                "launch_us_isolated_sinks_disabled": round(kern_none, 3)}

    def e2e(self, steps):
        """End to end through the public API: pinned host inputs -> device,
        the call, results -> host, each step on one of two streams in turn
        (its own device buffers), so that one step's copies overlap the other
        step's call and the copies in the other direction."""
        torch = self.torch
        nslot = 2
        ios = [self.r.host_io(k) for k in range(nslot)]
        host_in = [h.pin_memory() for h in ios[0][0]]
        dev_in = [[torch.empty_like(h, device="cuda") for h in host_in] for _ in range(nslot)]
        host_out = [[torch.empty_like(o, device="cpu").pin_memory() for o in io[1]]
                    for io in ios]
        streams = [torch.cuda.Stream() for _ in range(nslot)]

        def step(i):
            k = i % nslot
            with torch.cuda.stream(streams[k]):
                for d_, h_ in zip(dev_in[k], host_in):
                    d_.copy_(h_, non_blocking=True)
                ios[k][2](dev_in[k])
                for h_, o_ in zip(host_out[k], ios[k][1]):
                    h_.copy_(o_, non_blocking=True)

        for i in range(2 * nslot):
            step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()
        self.barrier()
        e0.record(cur)
        for s_ in streams:
            s_.wait_event(e0)
        for i in range(steps):
            step(i)
        for s_ in streams:
            cur.wait_stream(s_)
        e1.record(cur)
        self.barrier()
        ms = max_over_ranks(e0.elapsed_time(e1), self.dist, "cuda")
        h2d = sum(h.numel() * h.element_size() for h in host_in)
        d2h = sum(h.numel() * h.element_size() for h in host_out[0])
        return {"value": round(ms * 1000.0 / steps / self.world, 2), "unit": "us/call",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    def sustained(self, seconds):
        """Back-to-back calls for about ``seconds`` (a count taken from a
        short probe), timed as one region: the per-call time with the GPU
        held busy long enough for its clocks and power to settle."""
        probe = max(self.timed(self.r.mode, 200) / 200.0, 1e-3)
        n = int(max(200, seconds * 1e3 / probe))
        ms = self.timed(self.r.mode, n)
        return {"value": round(ms * 1000.0 / n / self.world, 3), "unit": "us/call",
                "calls": n, "seconds": round(ms / 1000.0, 3)}

    def roofline(self, call_us, traffic, src_hash):
        hbm_peak, tf_peak, peak_src = measured_peaks()
        gbs = self.nbytes / (call_us * 1e-6) / 1e9
        tfs = self.flops / (call_us * 1e-6) / 1e12
        if self.r.bound == "tensor":
            roof = {"bound": "tensor", "achieved": round(tfs, 1), "peak": tf_peak,
                    "unit": "TFLOP/s", "frac": round(tfs / tf_peak, 4), "traffic": traffic}
            other = {"alg_gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / hbm_peak, 4)}
        else:
            roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": traffic}
            other = {"alg_tflops": round(tfs, 2),
                     "frac_of_bf16_peak": round(tfs / tf_peak, 4)}
        roof.update({"peak_source": peak_src, "alg_bytes": self.nbytes,
                     "alg_flops": self.flops, "call_us": round(call_us, 3),
                     "source_hash": src_hash})
        return roof, other


def workload_entry(name, steps, dist, world, e2e_steps):
    """One configuration of the workload set, measured with the contract's
    rules on its own inputs: its per-call time and roofline, sink cost,
    isolated launch and end-to-end time."""
    import torch
    runner = RUNNERS[name](name)
    b = Bench(runner, dist, world)
    b.warm(max(10, steps // 10))
    ms = b.timed(runner.mode, steps)
    call_us = ms * 1000.0 / steps
    src_hash = kernel_source_hash(runner.source)
    roof, other = b.roofline(call_us, recorded_traffic(name, src_hash), src_hash)
    sc = b.sink_cost(max(steps // 2, 40))
    roof["launch_us_isolated"] = sc.pop("launch_us_isolated")
    entry = {"value": round(call_us / world, 3), "unit": "us/call", "steps": steps,
             "roofline": roof, "secondary": other, "e2e": b.e2e(max(10, e2e_steps // 2)),
             "gpu_launches": steps * runner.launches_per_call(),
             "config": arm_config(runner, world)}
    entry.update(sc)
    if name in PAGES_H100_US:
        entry["vs_pages_h100"] = round(entry["value"] / PAGES_H100_US[name], 4)
    del b, runner
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="vision_window_16384tok", choices=sorted(RUNNERS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure only --workload (no per-configuration entries)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--only-timed", action="store_true",
                    help="warm-up and the timed region only (for profiler launch lists): no "
                         "sink-cost, isolated-launch, end-to-end, sustained or per-workload legs")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.steps is None:
        args.steps = 500 if args.workload.startswith("dsa_block_prefill") else 5000

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    runner = RUNNERS[args.workload](args.workload)
    b = Bench(runner, dist, world)
    # the clocks are sampled over every timed leg of the run
    sampler = ClockSampler(gpu_uuid())
    b.warm(args.warmup)
    step_ms = b.timed(runner.mode, args.steps) / args.steps
    call_us = step_ms * 1000.0
    if args.only_timed:
        sc = {"sink_cost": None, "sink_cost_isolated": None, "launch_us_isolated": None,
              "launch_us_isolated_sinks_disabled": None}
        e2e = sustained = None
    else:
        sc = b.sink_cost(args.steps)
        e2e = b.e2e(args.e2e_steps)
        sustained = b.sustained(SUSTAINED_S)

    src_hash = kernel_source_hash(runner.source)
    traffic = recorded_traffic(args.workload, src_hash)
    roof, other = b.roofline(call_us, traffic, src_hash)
    roof["launch_us_isolated"] = sc["launch_us_isolated"]
    roof["sustained_call_us"] = sustained["value"] if sustained else None

    workloads = {}
    if not (args.no_workloads or args.only_timed) and args.workload == "vision_window_16384tok":
        del b
        torch.cuda.empty_cache()
        for name, steps in EXTRA_WORKLOADS:
            try:
                workloads[name] = workload_entry(name, steps, dist, world, args.e2e_steps)
            except Exception as exc:  # reported, never hidden
                workloads[name] = {"error": "%s: %s" % (type(exc).__name__, exc)}
            log("workload %s: %s" % (name, json.dumps(workloads[name].get("value"))))
    clocks = sampler.stop()

    import attention_head_sinks_gb300 as sa
    err = sa.sa_device_error()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    value_us = job_value_us(step_ms, world)
    head = {"value": round(value_us, 3), "unit": "us/call", "steps": args.steps,
            "roofline": roof, "sink_cost": sc["sink_cost"], "e2e": e2e,
            "gpu_launches": args.steps * runner.launches_per_call()}
    if workloads:
        workloads = dict([(args.workload, head)] + list(workloads.items()))
    line = {
        "metric": METRIC,
        "value": round(value_us, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": (round(value_us / PAGES_H100_US[args.workload], 4)
                        if args.workload in PAGES_H100_US else None),
        "dtype": "bf16",
        "data": "synthetic",
        "config": arm_config(runner, world),
        "roofline": roof,
        "secondary": other,
        "sink_cost": sc["sink_cost"],
        "sink_cost_isolated": sc["sink_cost_isolated"],
        "launch_us_isolated_sinks_disabled": sc["launch_us_isolated_sinks_disabled"],
        "sustained": sustained,
        "e2e": e2e,
        "gpu_launches": args.steps * runner.launches_per_call(),
        "clocks": clocks,
        "device_error": err,
    }
    if workloads:
        line["workloads"] = workloads
    if not (args.no_cpu_baseline or args.only_timed):
        line["cpu_baseline"] = cpu_baseline(runner)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
