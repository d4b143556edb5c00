"""Drives the library through its public API on the synthetic workloads.

Used by the benchmark and the GPU tests: it allocates pools and buffers with
PyTorch, fills caches through ``kv_append``, runs decode steps, the
serving-mix allocation protocol on the library's own block pool, and the
prefill-then-decode flow.  Every step calls the C ABI; nothing here computes
attention or slots itself.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (KvcConfig, kv_append, kv_block_alloc, kv_block_release, kv_block_share, kv_cache_create,
               kv_cache_destroy, kv_copy_blocks, kvc_copy_async, kv_slot_mapping, kv_step_prepare,
               paged_decode_append_attention, paged_decode_attention, paged_decode_plan, paged_decode_workspace_init,
               prefill_attention)

F16_NAN = 0x7E00  # a quiet-NaN bit pattern used to poison cache slots nobody owns


def _dev(a, device, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def poisoned_pool(shape, device) -> torch.Tensor:
    """fp16 pool filled with NaN bits: any read of a slot outside a context would show up."""
    return torch.full(shape, F16_NAN, dtype=torch.int16, device=device).view(torch.float16)


class DecodeSession:
    """A paged cache holding a DecodeWorkload's history, ready for decode steps on every layer."""

    def __init__(self, wl, device="cuda", out_dtype=torch.float32, blocks_per_split=0, poison=True):
        self.wl = wl
        self.device = device
        cfg = KvcConfig(num_layers=wl.L, num_blocks=wl.NB, num_kv_heads=wl.Hkv, head_dim=wl.D, block_size=wl.bs)
        self.cfg = cfg
        alloc = poisoned_pool if poison else (lambda s, d: torch.zeros(s, dtype=torch.float16, device=d))
        self.k_pool = alloc(cfg.pool_shape, device)
        self.v_pool = alloc(cfg.pool_shape, device)
        self.h = kv_cache_create(cfg, self.k_pool, self.v_pool)
        B = wl.B
        self.max_ctx = int(wl.ctx.max())
        self.block_table = _dev(wl.block_table, device)
        self.context_lens = _dev(wl.ctx, device)
        ones = np.ones(B, np.int32)
        self.hist_slots = _dev(kv_slot_mapping(wl.block_table, np.zeros(B, np.int32), wl.ctx - 1, wl.bs), device)
        self.step_slots_host = kv_slot_mapping(wl.block_table, wl.ctx - 1, ones, wl.bs)
        self.step_slots = _dev(self.step_slots_host, device)
        self.q = _dev(wl.q, device)
        self.k_new = _dev(wl.k_new, device)
        self.v_new = _dev(wl.v_new, device)
        self.out = torch.empty((wl.L, B, wl.Hq, wl.D), dtype=out_dtype, device=device)
        self.blocks_per_split = blocks_per_split
        self.nsplit, self.bps, ws = paged_decode_plan(B, wl.Hq, wl.Hkv, wl.D, self.max_ctx, blocks_per_split)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        paged_decode_workspace_init(self.workspace)

    def fill(self):
        """Write every sequence's history (positions 0 .. ctx-2) into the cache, layer by layer."""
        for layer in range(self.wl.L):
            kh = _dev(self.wl.k_hist[layer], self.device)
            vh = _dev(self.wl.v_hist[layer], self.device)
            kv_append(self.h, layer, kh, vh, self.hist_slots)
        return self

    def append(self, layer, stream=None):
        kv_append(self.h, layer, self.k_new[layer], self.v_new[layer], self.step_slots, stream=stream)

    def decode(self, layer, stream=None):
        paged_decode_attention(self.q[layer], self.k_pool[layer], self.v_pool[layer], self.block_table,
                               self.context_lens, self.wl.scale, self.out[layer], self.workspace, self.max_ctx,
                               self.blocks_per_split, stream=stream)

    def decode_append(self, layer, stream=None):
        """Fused append + decode of one layer."""
        paged_decode_append_attention(self.q[layer], self.k_new[layer], self.v_new[layer], self.k_pool[layer],
                                      self.v_pool[layer], self.block_table, self.context_lens, self.wl.scale,
                                      self.out[layer], self.workspace, self.max_ctx, self.blocks_per_split,
                                      stream=stream)

    def step(self, stream=None, fused=False):
        """One decode step: for every layer, append the new token's K/V, then attend.

        fused=False: kv_append then paged_decode_attention; fused=True: paged_decode_append_attention."""
        for layer in range(self.wl.L):
            if fused:
                self.decode_append(layer, stream)
            else:
                self.append(layer, stream)
                self.decode(layer, stream)

    def capture(self, fused=True, decode_only=False, stream=None):
        """CUDA graph of one step (or of the 24 decode calls alone); eager warm-up first."""
        stream = stream or torch.cuda.Stream(self.device)
        with torch.cuda.stream(stream):
            self._graph_body(fused, decode_only)
        torch.cuda.synchronize(self.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self._graph_body(fused, decode_only)
        torch.cuda.synchronize(self.device)
        return graph

    def _graph_body(self, fused, decode_only):
        if decode_only:
            for layer in range(self.wl.L):
                self.decode_append(layer) if fused else self.decode(layer)
        else:
            self.step(fused=fused)

    def close(self):
        if self.h:
            kv_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def serving_mix(mix, device="cuda", out_dtype=torch.float32, poison=True):
    """The serving-mix protocol on the library's block pool: groups of `mix.group` sequences share the blocks of a
    common prompt prefix (refcounted, allocated once per group), each sequence owns the blocks of its private
    tail, and one decode step appends a token per sequence — a sequence whose last block is shared gets a
    private copy first (copy-on-write) — and then runs paged decode over the new tables.

    Returns a dict: block tables before/after the step, copy pairs, slots, pools and the output."""
    bs = mix.bs
    cfg = KvcConfig(num_layers=1, num_blocks=mix.NB, num_kv_heads=mix.Hkv, head_dim=mix.D, block_size=bs)
    alloc = poisoned_pool if poison else (lambda s, d: torch.zeros(s, dtype=torch.float16, device=d))
    k_pool, v_pool = alloc(cfg.pool_shape, device), alloc(cfg.pool_shape, device)
    h = kv_cache_create(cfg, k_pool, v_pool)
    try:
        for _ in range(mix.NB):
            kv_block_alloc(h)
        for pid in mix.free_order:
            kv_block_release(h, int(pid))
        B, G = mix.B, mix.group
        npre = -(-mix.prefix_len // bs)
        tables = [[] for _ in range(B)]
        for g in range(-(-B // G)):
            members = range(g * G, min(B, (g + 1) * G))
            prefix_pages = [kv_block_alloc(h) for _ in range(npre)]
            for b in members:
                need = -(-min(mix.prefix_len, int(mix.ctx[b]) - 1) // bs)
                for pid in prefix_pages[:need]:
                    kv_block_share(h, pid)
                tables[b] = list(prefix_pages[:need])
            n_pre = max(min(mix.prefix_len, int(mix.ctx[b]) - 1) for b in members)
            slots = kv_slot_mapping(np.array([prefix_pages], np.int32), [0], [n_pre], bs)
            kv_append(h, 0, _dev(mix.prefix_k[g, :n_pre], device), _dev(mix.prefix_v[g, :n_pre], device),
                      _dev(slots, device))
            for pid in prefix_pages:
                kv_block_release(h, pid)
            for b in members:
                while len(tables[b]) * bs < int(mix.ctx[b]) - 1:
                    tables[b].append(kv_block_alloc(h))
                n_suf = int(mix.suffix_off[b + 1] - mix.suffix_off[b])
                if n_suf:
                    row = np.array([tables[b]], np.int32)
                    slots = kv_slot_mapping(row, [mix.prefix_len], [n_suf], bs)
                    sl = slice(int(mix.suffix_off[b]), int(mix.suffix_off[b + 1]))
                    kv_append(h, 0, _dev(mix.suffix_k[sl], device), _dev(mix.suffix_v[sl], device),
                              _dev(slots, device))
        tables_before = [list(t) for t in tables]
        mb = max(-(-int(c) // bs) for c in mix.ctx)
        table = np.full((B, mb), -1, np.int32)
        nblk = np.zeros(B, np.int32)
        for b in range(B):
            table[b, :len(tables[b])] = tables[b]
            nblk[b] = len(tables[b])
        slots, copies = kv_step_prepare(h, table, nblk, mix.ctx - 1)
        kv_copy_blocks(h, copies[:, 0], copies[:, 1])
        kv_append(h, 0, _dev(mix.k_new, device), _dev(mix.v_new, device), _dev(slots, device))
        q = _dev(mix.q, device)
        out = torch.empty((B, mix.Hq, mix.D), dtype=out_dtype, device=device)
        max_ctx = int(mix.ctx.max())
        _, _, ws = paged_decode_plan(B, mix.Hq, mix.Hkv, mix.D, max_ctx)
        workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        paged_decode_workspace_init(workspace)
        paged_decode_attention(q, k_pool[0], v_pool[0], _dev(table, device), _dev(mix.ctx, device), mix.scale, out,
                               workspace, max_ctx)
        torch.cuda.synchronize()
        return {"tables_before": tables_before, "block_table": table, "copies": copies, "slots": slots,
                "k_cache": k_pool[0], "v_cache": v_pool[0], "out": out, "handle": None}
    finally:
        kv_cache_destroy(h)


def prefill_then_decode(wl, causal=True, device="cuda", out_dtype=torch.float32, poison=True):
    """Prefill a packed batch, write all its K/V into a paged cache, then one decode token per sequence."""
    q, k, v = _dev(wl.q, device), _dev(wl.k, device), _dev(wl.v, device)
    cu = _dev(wl.cu_seqlens, device)
    T = q.shape[0]
    out = torch.empty((T, wl.Hq, wl.D), dtype=out_dtype, device=device)
    prefill_attention(q, k, v, cu, max(wl.seqlens), wl.scale, causal, out)
    n = len(wl.seqlens)
    cfg = KvcConfig(num_layers=1, num_blocks=wl.NB, num_kv_heads=wl.Hkv, head_dim=wl.D, block_size=wl.bs)
    alloc = poisoned_pool if poison else (lambda s, d: torch.zeros(s, dtype=torch.float16, device=d))
    k_pool, v_pool = alloc(cfg.pool_shape, device), alloc(cfg.pool_shape, device)
    h = kv_cache_create(cfg, k_pool, v_pool)
    try:
        seqlens = np.array(wl.seqlens, np.int32)
        slots = kv_slot_mapping(wl.block_table, np.zeros(n, np.int32), seqlens, wl.bs)
        kv_append(h, 0, k, v, _dev(slots, device))
        step = kv_slot_mapping(wl.block_table, seqlens, np.ones(n, np.int32), wl.bs)
        kv_append(h, 0, _dev(wl.k_dec, device), _dev(wl.v_dec, device), _dev(step, device))
        ctx = seqlens + 1
        dec = torch.empty((n, wl.Hq, wl.D), dtype=out_dtype, device=device)
        _, _, ws = paged_decode_plan(n, wl.Hq, wl.Hkv, wl.D, int(ctx.max()))
        workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        paged_decode_workspace_init(workspace)
        paged_decode_attention(_dev(wl.q_dec, device), k_pool[0], v_pool[0], _dev(wl.block_table, device),
                               _dev(ctx, device), wl.scale, dec, workspace, int(ctx.max()))
        torch.cuda.synchronize()
        return {"prefill_out": out, "decode_out": dec, "k_cache": k_pool[0], "v_cache": v_pool[0]}
    finally:
        kv_cache_destroy(h)


def _align16(n: int) -> int:
    return (n + 15) & ~15


class HostStep:
    """A DecodeSession's step fed from pinned host memory, its output returned there, with the copies overlapped
    with the calls as a serving loop whose inputs arrive from the host would run it.

    The step's inputs sit in one pinned host buffer: a header (block table, context lengths, append slots),
    then per layer that layer's q, k_new and v_new, each 16-byte aligned.  A device buffer has the same layout
    and every call receives views into it.  Every copy is a staging copy (kvc_copy_async: a kernel that reads or
    writes the pinned buffer over the host link) in the stream's kernel sequence.  In: the header with layers 0
    and 1 before layer 0's call; the later layers ahead, in pieces of growing size, each alongside an earlier
    layer's call (layers 2-3 alongside layer 0's, 4-7 alongside layer 1's, the rest alongside layer 3's; one
    piece for all of them made layer 1 wait for it).  Out: the outputs of layers
    [lo, hi) ahead, alongside layer hi's call (a decode call lets the next kernel start only once the calls before
    it have finished, so those outputs are final), eight layers at a time; the last layer's after its call.
    Every call is checked and converted once, at construction (the prepare=True form of the API)."""

    GROUP = 8  # layers per device-to-host copy

    def __init__(self, sess: DecodeSession):
        wl, dev = sess.wl, sess.device
        self.sess, self.device, self.L = sess, dev, wl.L
        parts = [("block_table", np.ascontiguousarray(wl.block_table, np.int32)),
                 ("context_lens", np.ascontiguousarray(wl.ctx, np.int32)),
                 ("slots", np.ascontiguousarray(sess.step_slots_host, np.int64))]
        for layer in range(wl.L):
            parts += [(("q", layer), np.ascontiguousarray(wl.q[layer], np.float16)),
                      (("k_new", layer), np.ascontiguousarray(wl.k_new[layer], np.float16)),
                      (("v_new", layer), np.ascontiguousarray(wl.v_new[layer], np.float16))]
        offs, pos, layer_end = {}, 0, []
        for name, a in parts:
            offs[name] = pos
            pos = _align16(pos + a.nbytes)
            if name[0] == "v_new":
                layer_end.append(pos)
        self.h_buf = torch.empty(pos, dtype=torch.uint8).pin_memory()
        hb = self.h_buf.numpy()
        hb[:] = 0
        for name, a in parts:
            hb[offs[name]:offs[name] + a.nbytes] = a.reshape(-1).view(np.uint8)
        self.d_buf = torch.zeros(pos, dtype=torch.uint8, device=dev)
        tdt = {np.dtype(np.int32): torch.int32, np.dtype(np.int64): torch.int64, np.dtype(np.float16): torch.float16}

        def view(name, a):
            return self.d_buf[offs[name]:offs[name] + a.nbytes].view(tdt[a.dtype]).view(a.shape)
        arrays = dict(parts)
        self.block_table, self.context_lens, self.slots = (view(n, arrays[n])
                                                          for n in ("block_table", "context_lens", "slots"))
        self.q, self.k_new, self.v_new = ([view((n, layer), arrays[(n, layer)]) for layer in range(wl.L)]
                                          for n in ("q", "k_new", "v_new"))
        self.k_pool = [sess.k_pool[layer] for layer in range(wl.L)]
        self.v_pool = [sess.v_pool[layer] for layer in range(wl.L)]
        self.out = [sess.out[layer] for layer in range(wl.L)]
        self.h_out = torch.empty(sess.out.shape, dtype=sess.out.dtype).pin_memory()
        self.h_out_layers = [self.h_out[layer] for layer in range(wl.L)]
        cut = layer_end[min(1, wl.L - 1)]  # header + layers 0 and 1
        self.first = (self.d_buf[:cut], self.h_buf[:cut])
        # layers [a, b) staged ahead alongside layer a / 2 - 1's call
        starts = [a for a in (2, 4, 8) if a < wl.L]
        self.ahead_in = {}
        for i, a in enumerate(starts):
            b = starts[i + 1] if i + 1 < len(starts) else wl.L
            lo, hi = layer_end[a - 1], layer_end[b - 1]
            self.ahead_in[a // 2 - 1] = (self.d_buf[lo:hi], self.h_buf[lo:hi])
        # device-to-host groups [lo, hi) of all layers but the last, each sent alongside layer hi's call
        self.groups = {min(g + self.GROUP, wl.L - 1): (self.h_out[g:min(g + self.GROUP, wl.L - 1)],
                                                       sess.out[g:min(g + self.GROUP, wl.L - 1)])
                       for g in range(0, wl.L - 1, self.GROUP)}
        self.h2d_bytes = pos
        self.d2h_bytes = self.h_out.numel() * self.h_out.element_size()
        # every call of the step checked and converted once (PreparedCall); run() only launches them
        self._first = kvc_copy_async(*self.first, prepare=True)
        self._ahead_in = {k: kvc_copy_async(*v, ahead=True, prepare=True) for k, v in self.ahead_in.items()}
        self._groups = {k: kvc_copy_async(*v, ahead=True, prepare=True) for k, v in self.groups.items()}
        self._last = kvc_copy_async(self.h_out_layers[-1], self.out[-1], prepare=True)
        self._fused = [paged_decode_append_attention(self.q[layer], self.k_new[layer], self.v_new[layer],
                                                     self.k_pool[layer], self.v_pool[layer], self.block_table,
                                                     self.context_lens, wl.scale, self.out[layer], sess.workspace,
                                                     sess.max_ctx, sess.blocks_per_split, prepare=True)
                       for layer in range(wl.L)]
        self._unfused = [(kv_append(sess.h, layer, self.k_new[layer], self.v_new[layer], self.slots, prepare=True),
                          paged_decode_attention(self.q[layer], self.k_pool[layer], self.v_pool[layer],
                                                 self.block_table, self.context_lens, wl.scale, self.out[layer],
                                                 sess.workspace, sess.max_ctx, sess.blocks_per_split, prepare=True))
                         for layer in range(wl.L)]

    def run(self, fused=True):
        """One step on the current stream: copies in, every layer's call(s), copies out (all asynchronous)."""
        cs = torch.cuda.current_stream(self.device)
        self._first(cs)
        for layer in range(self.L):
            if fused:
                self._fused[layer](cs)
            else:
                append, decode = self._unfused[layer]
                append(cs)
                decode(cs)
            if layer in self._ahead_in:
                self._ahead_in[layer](cs)
            if layer in self._groups:
                self._groups[layer](cs)
        self._last(cs)
