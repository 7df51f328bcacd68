"""One FAST-AR attention layer on one GPU: cache state, the per-chunk step, and the
dense baseline, all driven through libfastar's C ABI.

PyTorch only supplies device memory, streams, events and CUDA graphs; every stage
of the step runs in libfastar's kernels (there is no fallback path: a missing
library raises).

The step for one chunk of Nq = F*Tf tokens (FAST-AR technical summary §2.A–C):
  1. buckets of the queries (top-r) and of the current keys (argmax, plus |k|)
  2. TempCache top-1 match of every query against the cache -> eviction flags
  3. compaction into the other half of a double-buffered cache (FIFO cap M)
  4. counting sort of the cache keys and of the (query, slot) pairs by bucket
  5. AnnSA bucket-restricted self-attention -> o_self
  6. AnnCA prompt selection per latent frame
  7. cross-attention over the kept prompt tokens -> o_cross
Stages 6-7 depend only on stage 1, so they run on a second stream alongside 2-5.

merge=True runs the merge variant (technical summary §2.A, Theoretical Basis: Lemma
5.1): every cache entry carries a group count g; an evicted entry is folded into the
current entry that owns it (count-weighted mean value, summed count) instead of being
dropped, and AnnSA shifts every key's logit by ln g.

pq=(m, Kc) runs the quantization variant of the match (technical summary §2.A, "LSH or
Quantization"): every cache entry also carries its product-quantization code, the
current keys are encoded each step, and the match ranks the decoded cached keys.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import _lib as L


def _i32(*shape, dev):
    return torch.zeros(shape, dtype=torch.int32, device=dev)


def _f32(*shape, dev):
    return torch.zeros(shape, dtype=torch.float32, device=dev)


class CacheState:
    """One half of the double-buffered TempCache: rows, norms, buckets, lengths (and,
    for the merge variant, group counts)."""

    def __init__(self, H, M, d, dtype, dev, grouped=False, pq_m=0):
        self.k = torch.zeros((H, M, d), dtype=dtype, device=dev)
        self.v = torch.zeros((H, M, d), dtype=dtype, device=dev)
        self.knorm = _f32(H, M, dev=dev)
        self.kb = _i32(H, M, 1, dev=dev)
        self.len = _i32(H, dev=dev)
        self.g = _i32(H, M, dev=dev) if grouped else None
        self.codes = torch.zeros((H, M, pq_m), dtype=torch.uint8, device=dev) if pq_m else None

    def nbytes(self) -> int:
        ts = [self.k, self.v, self.knorm, self.kb, self.len] + [t for t in (self.g, self.codes) if t is not None]
        return sum(t.numel() * t.element_size() for t in ts)


class FastARLayer:
    """Device state and step of one FAST-AR attention layer (one head group, one GPU)."""

    def __init__(self, H: int, d: int, Tf: int, F: int, M: int, B: int, r: int, P: int, tau: float,
                 tau_ca: float, topk: int = 16, dtype: torch.dtype = torch.bfloat16, gate: bool = True,
                 device: str | torch.device = "cuda", scale: Optional[float] = None,
                 diagnostics: bool = False, merge: bool = False, pq: Optional[tuple] = None):
        """diagnostics=True also produces the second-best match cosine s2 (a slower
        match epilogue); the step's results are the same either way.  merge=True: the
        Lemma 5.1 merge variant (group counts, folded values, ln g logit shift).  pq=(m, Kc):
        the quantised match (set the codebooks with set_codebooks before loading a cache)."""
        L.load()
        if M < F * Tf:
            raise ValueError(f"cache cap M={M} must hold one chunk of {F * Tf} tokens")
        self.H, self.d, self.Tf, self.F, self.M, self.B, self.r, self.P = H, d, Tf, F, M, B, r, P
        self.Nq = F * Tf
        self.tau, self.tau_ca, self.topk, self.gate = float(tau), float(tau_ca), int(topk), bool(gate)
        self.diagnostics = bool(diagnostics)
        self.merge = bool(merge)
        self.pq = tuple(pq) if pq else None
        pq_m = self.pq[0] if self.pq else 0
        self.dtype = dtype
        self.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
        dev = torch.device(device)
        self.dev = dev
        Nq = self.Nq
        self.caches = [CacheState(H, M, d, dtype, dev, self.merge, pq_m), CacheState(H, M, d, dtype, dev, self.merge, pq_m)]
        self.cur = 0
        # prompt
        self.kp = torch.zeros((H, P, d), dtype=dtype, device=dev)
        self.vp = torch.zeros((H, P, d), dtype=dtype, device=dev)
        self.pb = _i32(H, P, 1, dev=dev)
        self.centroids = torch.zeros((H, B, d), dtype=dtype, device=dev)
        # per-step intermediates and outputs
        self.qb = _i32(H, Nq, r, dev=dev)
        self.kb_cur = _i32(H, Nq, 1, dev=dev)
        self.kcur_norm = _f32(H, Nq, dev=dev)
        self.qnorm = _f32(H, Nq, dev=dev)   # the queries' norms, written by the assignment for AnnCA
        self.top1 = _i32(H, Nq, dev=dev)
        self.s1 = _f32(H, Nq, dev=dev)
        self.s2 = _f32(H, Nq, dev=dev)
        self.evict = torch.zeros((H, M), dtype=torch.uint8, device=dev)
        self.owner = _i32(H, M, dev=dev) if (self.merge or pq) else None
        self.index_map = _i32(H, M, dev=dev)
        self.kperm = _i32(H, M, dev=dev)
        self.koff = _i32(H, B + 1, dev=dev)
        # the replace variant in bf16: the compaction also sorts the new cache's keys and
        # writes AnnSA's bucket-ordered copy of K/V as it moves the rows
        self.presort = dtype == torch.bfloat16 and not self.merge
        if self.presort:
            self.kpos = _i32(H, M, dev=dev)
            self.k_sorted = torch.zeros((H, M, d), dtype=dtype, device=dev)
            self.v_sorted = torch.zeros((H, M, d), dtype=dtype, device=dev)
        self.qperm = _i32(H, Nq * r, dev=dev)
        self.qoff = _i32(H, B + 1, dev=dev)
        self.o_self = torch.zeros((H, Nq, d), dtype=dtype, device=dev)
        self.lse_self = _f32(H, Nq, dev=dev)
        self.keep = torch.zeros((H, F, P), dtype=torch.uint8, device=dev)
        self.kidx = _i32(H, F, P, dev=dev)
        self.kcnt = _i32(H, F, dev=dev)
        self.score = _f32(H, F, P, dev=dev)
        self.o_cross = torch.zeros((H, Nq, d), dtype=dtype, device=dev)
        self.lse_cross = _f32(H, Nq, dev=dev)
        self.dev_status = _i32(1, dev=dev)

        def ws(op, **kw):
            nbytes = L.workspace_bytes(op, H, **kw)
            return torch.zeros(max(16, (nbytes + 15) // 16 * 16), dtype=torch.uint8, device=dev)

        self.ws_match = ws(L.OP_MATCH, n=Nq, M=M, d=d)
        self.ws_attn = ws(L.OP_SPARSE_ATTN, n=Nq, M=M, d=d, B=B, r=r)
        # bf16: the selection's ranking launch copies the kept prompt rows into per-frame
        # planes, which the cross-attention reads as tiles (no gather launch of its own)
        self.kept = dtype == torch.bfloat16 and P > 0
        self.ws_cross = ws(L.OP_CROSS_ATTN, n=0, d=d, P=P, F=F) if P > 0 and not self.kept else None
        if self.kept:
            self.kp_kept = torch.zeros((H, F, P, d), dtype=dtype, device=dev)
            self.vp_kept = torch.zeros((H, F, P, d), dtype=dtype, device=dev)
        if self.pq:
            m, Kc = self.pq
            self.codebooks = torch.zeros((H, m, Kc, d // m), dtype=dtype, device=dev)
            self.codes_cur = torch.zeros((H, Nq, m), dtype=torch.uint8, device=dev)
            self.ws_match_pq = ws(L.OP_MATCH_PQ, n=Nq, M=M, d=d)
        self.side = torch.cuda.Stream(device=dev)
        self.mside = torch.cuda.Stream(device=dev)
        self.match_first = True
        self._graph = None
        self._graph_dir = None

    # ---- state ------------------------------------------------------------------------------
    @property
    def cache(self) -> CacheState:
        return self.caches[self.cur]

    def device_bytes(self) -> int:
        """Bytes of every device buffer the layer holds (constant over a rollout)."""
        tot = sum(c.nbytes() for c in self.caches)
        for t in vars(self).values():
            if isinstance(t, torch.Tensor):
                tot += t.numel() * t.element_size()
        return tot

    def set_centroids(self, C: torch.Tensor):
        self.centroids.copy_(C)

    def set_codebooks(self, cb: torch.Tensor):
        """Product-quantization codebooks [H, m, Kc, d/m] (quantised-match mode)."""
        self.codebooks.copy_(cb)

    def set_prompt(self, kp: torch.Tensor, vp: torch.Tensor):
        """Installs the prompt and assigns its key buckets (once per rollout)."""
        self.kp.copy_(kp)
        self.vp.copy_(vp)
        if self.P:
            L.fastar_bucket_assign(self.kp, self.centroids, 1, self.pb)

    def load_cache(self, k: torch.Tensor, v: torch.Tensor, g: Optional[torch.Tensor] = None):
        """Installs n raw entries (oldest first) as the current cache: norms and key
        buckets are computed by the library.  g: group counts [H, n] (merge variant;
        default 1 each)."""
        n = k.shape[1]
        if n > self.M:
            raise ValueError("more entries than the cache cap")
        c = self.cache
        c.k[:, :n].copy_(k)
        c.v[:, :n].copy_(v)
        if n:
            kb = _i32(self.H, n, 1, dev=self.dev)
            kn = _f32(self.H, n, dev=self.dev)
            L.fastar_bucket_assign(c.k[:, :n], self.centroids, 1, kb, None, kn)
            c.kb[:, :n].copy_(kb)
            c.knorm[:, :n].copy_(kn)
        if c.codes is not None and n:
            codes = torch.zeros((self.H, n, self.pq[0]), dtype=torch.uint8, device=self.dev)
            L.fastar_pq_encode(c.k[:, :n], self.codebooks, codes)   # [H, n, m], contiguous
            c.codes[:, :n].copy_(codes)
        if c.g is not None:
            if g is None:
                c.g[:, :n].fill_(1)
            else:
                c.g[:, :n].copy_(g)
        c.len.fill_(n)

    def reset(self):
        for c in self.caches:
            c.len.zero_()
        self.cur = 0

    # ---- the step ------------------------------------------------------------------------------
    def _enqueue(self, q, k_cur, v_cur, src: int, timer=None, serial: bool = False):
        """Enqueues one step reading cache `src` and writing cache 1 - src.

        timer: optional callable(name, stream, phase) invoked around each stage
        ("begin"/"end") on the stream the stage is launched on (for per-stage timing
        with CUDA events; never used inside a graph capture).
        serial: run the AnnCA branch on the main stream too (one kernel at a time,
        so that per-stage times are those of each stage alone)."""
        cin, cout = self.caches[src], self.caches[1 - src]
        main = torch.cuda.current_stream(self.dev)
        side = main if serial else self.side
        t = timer or (lambda *a: None)

        def match(stream):
            t("tempcache_match", stream, "begin")
            if self.pq:
                L.fastar_tempcache_match_pq(q, k_cur, cin.k, cin.knorm, cin.codes, cin.len, self.codebooks,
                                            self.tau, self.top1, self.s1, self.evict, self.dev_status,
                                            self.ws_match_pq, owner=self.owner)
            else:
                L.fastar_tempcache_match(q, k_cur, cin.k, cin.knorm, cin.len, self.tau, self.top1, self.s1,
                                         self.s2 if self.diagnostics else None,
                                         self.evict, self.dev_status, self.ws_match, owner=self.owner)
            t("tempcache_match", stream, "end")

        # the match needs only the step's inputs and the incoming cache: it starts at once
        # on its own stream, beside the bucket assignment, the pair sort and AnnCA
        early = self.match_first and not serial
        if early:
            ev0 = torch.cuda.Event()
            ev0.record(main)
            self.mside.wait_event(ev0)
            with torch.cuda.stream(self.mside):
                match(self.mside)
            evm = torch.cuda.Event()
            evm.record(self.mside)
        t("bucket_assign", main, "begin")
        L.fastar_bucket_assign_qk(q, k_cur, self.centroids, self.r, self.qb, self.kb_cur, self.kcur_norm,
                                  q_norms=self.qnorm)
        t("bucket_assign", main, "end")
        if self.pq:
            t("pq_encode", main, "begin")
            L.fastar_pq_encode(k_cur, self.codebooks, self.codes_cur)
            t("pq_encode", main, "end")
        # the (query, slot) pairs by bucket: AnnSA's query-side order (the sorted compaction
        # writes it in its own planning launch; the other paths sort here, where AnnCA's
        # SIMT scorer can use it too)
        if not self.presort:
            t("bucket_sort_q", main, "begin")
            L.fastar_bucket_sort(self.qb, self.B, self.qperm, self.qoff, None, self.dev_status)
            t("bucket_sort_q", main, "end")
        # AnnCA branch on the side stream
        if not serial:
            ev = torch.cuda.Event()
            ev.record(main)
            side.wait_event(ev)
        with torch.cuda.stream(side):
            t("annca_select", side, "begin")
            self._annca(q, self.qperm if not self.presort else None, self.qoff if not self.presort else None,
                        self.qnorm)
            t("annca_select", side, "end")
            t("cross_attn_subset", side, "begin")
            self._cross(q, self.o_cross)
            t("cross_attn_subset", side, "end")
        # TempCache + AnnSA on the main stream
        if early:
            main.wait_event(evm)
        else:
            match(main)
        t("cache_compact", main, "begin")
        if self.merge:
            L.fastar_cache_compact_merge(k_cur, v_cur, self.kcur_norm, self.kb_cur, cin.k, cin.v, cin.knorm, cin.kb,
                                         cin.g, cin.len, self.evict, self.top1, self.owner, cout.k, cout.v,
                                         cout.knorm, cout.kb, cout.g, cout.len, self.index_map, self.dev_status)
        elif self.presort:
            L.fastar_cache_compact_sorted(k_cur, v_cur, self.kcur_norm, self.kb_cur, cin.k, cin.v, cin.knorm, cin.kb,
                                          cin.len, self.evict, cout.k, cout.v, cout.knorm, cout.kb, cout.len,
                                          self.index_map, self.B, self.kperm, self.koff, self.kpos, self.k_sorted,
                                          self.v_sorted, self.dev_status, qb=self.qb, qperm=self.qperm,
                                          qoff=self.qoff)
        else:
            L.fastar_cache_compact(k_cur, v_cur, self.kcur_norm, self.kb_cur, cin.k, cin.v, cin.knorm, cin.kb,
                                   cin.len, self.evict, cout.k, cout.v, cout.knorm, cout.kb, cout.len,
                                   self.index_map, self.dev_status)
        if self.pq:
            L.fastar_pq_gather_codes(cin.codes, cin.len, self.codes_cur, self.index_map, cout.len, cout.codes,
                                     self.dev_status)
        t("cache_compact", main, "end")
        if not self.presort:   # (the sorted compaction has grouped the keys already)
            t("bucket_sort", main, "begin")
            L.fastar_bucket_sort(cout.kb, self.B, self.kperm, self.koff, cout.len, self.dev_status)
            t("bucket_sort", main, "end")
        t("sparse_attn", main, "begin")
        if self.merge:
            L.fastar_sparse_attn_grouped(q, self.r, self.B, self.qperm, self.qoff, cout.k, cout.v, self.kperm,
                                         self.koff, cout.g, self.scale, self.o_self, self.lse_self, self.dev_status,
                                         self.ws_attn)
        elif self.presort:
            L.fastar_sparse_attn_presorted(q, self.r, self.B, self.qperm, self.qoff, cout.k, cout.v, self.kperm,
                                           self.koff, self.k_sorted, self.v_sorted, self.scale, self.o_self,
                                           self.lse_self, self.dev_status, self.ws_attn)
        else:
            L.fastar_sparse_attn(q, self.r, self.B, self.qperm, self.qoff, cout.k, cout.v, self.kperm, self.koff,
                                 self.scale, self.o_self, self.lse_self, self.dev_status, self.ws_attn)
        t("sparse_attn", main, "end")
        if not serial:
            ev2 = torch.cuda.Event()
            ev2.record(side)
            main.wait_event(ev2)

    # ---- the two halves of the step, for a transformer block that projects its own
    # cross-attention queries (the self step commits the cache only with advance=True) ----
    def step_self(self, q, k_cur, v_cur, out=None, advance: bool = True):
        """TempCache + AnnSA on the current stream: bucket assignment of q and k_cur, the
        match against the current cache, compaction into the other half, the bucket sorts
        and the bucket-restricted attention -> out ([H, Nq, d] view; default o_self)."""
        cin, cout = self.caches[self.cur], self.caches[1 - self.cur]
        o = self.o_self if out is None else out
        L.fastar_bucket_assign_qk(q, k_cur, self.centroids, self.r, self.qb, self.kb_cur, self.kcur_norm)
        if not self.presort:
            L.fastar_bucket_sort(self.qb, self.B, self.qperm, self.qoff, None, self.dev_status)
        L.fastar_tempcache_match(q, k_cur, cin.k, cin.knorm, cin.len, self.tau, self.top1, self.s1, None,
                                 self.evict, self.dev_status, self.ws_match)
        if self.presort:
            L.fastar_cache_compact_sorted(k_cur, v_cur, self.kcur_norm, self.kb_cur, cin.k, cin.v, cin.knorm, cin.kb,
                                          cin.len, self.evict, cout.k, cout.v, cout.knorm, cout.kb, cout.len,
                                          self.index_map, self.B, self.kperm, self.koff, self.kpos, self.k_sorted,
                                          self.v_sorted, self.dev_status, qb=self.qb, qperm=self.qperm,
                                          qoff=self.qoff)
            L.fastar_sparse_attn_presorted(q, self.r, self.B, self.qperm, self.qoff, cout.k, cout.v, self.kperm,
                                           self.koff, self.k_sorted, self.v_sorted, self.scale, o, self.lse_self,
                                           self.dev_status, self.ws_attn)
        else:
            L.fastar_cache_compact(k_cur, v_cur, self.kcur_norm, self.kb_cur, cin.k, cin.v, cin.knorm, cin.kb,
                                   cin.len, self.evict, cout.k, cout.v, cout.knorm, cout.kb, cout.len,
                                   self.index_map, self.dev_status)
            L.fastar_bucket_sort(cout.kb, self.B, self.kperm, self.koff, cout.len, self.dev_status)
            L.fastar_sparse_attn(q, self.r, self.B, self.qperm, self.qoff, cout.k, cout.v, self.kperm, self.koff,
                                 self.scale, o, self.lse_self, self.dev_status, self.ws_attn)
        if advance:
            self.cur = 1 - self.cur
        return o

    def step_cross(self, q, out=None):
        """AnnCA on the current stream for its own queries q: their buckets, the
        frame-relevant prompt tokens, cross-attention over them -> out (default o_cross)."""
        o = self.o_cross if out is None else out
        L.fastar_bucket_assign(q, self.centroids, self.r, self.qb, None, self.qnorm)
        # the bf16 scorer masks dense tiles with qb itself; the bucket order helps the SIMT one
        order = q.dtype != torch.bfloat16
        if order:
            L.fastar_bucket_sort(self.qb, self.B, self.qperm, self.qoff, None, self.dev_status)
        self._annca(q, self.qperm if order else None, self.qoff if order else None, self.qnorm)
        self._cross(q, o)
        return o

    def _annca(self, q, qperm, qoff, qnorm=None):
        """The prompt selection for queries q (and, in bf16, the kept rows' planes); qnorm:
        q's norms as the bucket assignment wrote them."""
        kw = dict(vp=self.vp, kp_kept=self.kp_kept, vp_kept=self.vp_kept) if self.kept else {}
        L.fastar_annca_select(q, self.F, self.qb, self.kp, self.pb, self.tau_ca, self.topk, self.gate, self.keep,
                              self.kidx, self.kcnt, self.score, B=self.B, qperm=qperm, qoff=qoff, q_norms=qnorm,
                              **kw)

    def _cross(self, q, o):
        """Cross-attention of q over the kept prompt tokens -> o."""
        if self.kept:
            L.fastar_cross_attn_kept(q, self.F, self.kp_kept, self.vp_kept, self.kcnt, self.scale, o, self.lse_cross)
        else:
            L.fastar_cross_attn_subset(q, self.F, self.kp, self.vp, self.kidx, self.kcnt, self.scale, o,
                                       self.lse_cross, workspace=self.ws_cross)

    def step(self, q, k_cur, v_cur, advance: bool = True, timer=None, serial: bool = False):
        """Runs one chunk step (asynchronously, on the current stream).  With
        advance=False the cache state is not swapped, so the same step can be repeated;
        serial=True keeps every kernel on the current stream."""
        self._enqueue(q, k_cur, v_cur, self.cur, timer, serial)
        if advance:
            self.cur = 1 - self.cur
        return self.o_self, self.o_cross

    # ---- CUDA graph of one step ----------------------------------------------------------------
    def capture(self, q, k_cur, v_cur):
        """Captures one step (reading the current cache half) into a CUDA graph; the
        graph reads q/k_cur/v_cur from these exact tensors."""
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            self._enqueue(q, k_cur, v_cur, self.cur)     # warm-up outside capture
        torch.cuda.synchronize(self.dev)
        with torch.cuda.graph(g, stream=s):
            self._enqueue(q, k_cur, v_cur, self.cur)
        torch.cuda.synchronize(self.dev)
        self._graph, self._graph_dir = g, self.cur
        return g

    def replay(self):
        self._graph.replay()

    def status(self) -> int:
        return int(self.dev_status.item())


class DenseLayer:
    """The dense baseline: an append-only cache and full attention over it, plus
    cross-attention over the whole prompt."""

    def __init__(self, H, d, Nq, cap, P, dtype=torch.bfloat16, device="cuda", scale=None):
        L.load()
        dev = torch.device(device)
        self.H, self.d, self.Nq, self.cap, self.P = H, d, Nq, cap, P
        self.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
        self.k = torch.zeros((H, cap, d), dtype=dtype, device=dev)
        self.v = torch.zeros((H, cap, d), dtype=dtype, device=dev)
        self.kp = torch.zeros((H, P, d), dtype=dtype, device=dev)
        self.vp = torch.zeros((H, P, d), dtype=dtype, device=dev)
        self.n = 0
        self.o_self = torch.zeros((H, Nq, d), dtype=dtype, device=dev)
        self.o_cross = torch.zeros((H, Nq, d), dtype=dtype, device=dev)
        self.lse_self = _f32(H, Nq, dev=dev)
        self.lse_cross = _f32(H, Nq, dev=dev)

    def load_history(self, k, v):
        n = k.shape[1]
        self.k[:, :n].copy_(k)
        self.v[:, :n].copy_(v)
        self.n = n

    def set_prompt(self, kp, vp):
        self.kp.copy_(kp)
        self.vp.copy_(vp)

    def step_self(self, q, k_cur, v_cur, out=None, advance: bool = True):
        """Appends the chunk (at the current length; committed with advance=True) and
        attends over every key so far -> out ([H, Nq, d] view; default o_self)."""
        o = self.o_self if out is None else out
        nq = q.shape[1]
        L.fastar_dense_append(k_cur, v_cur, self.k, self.v, self.n)
        L.fastar_dense_attn(q, self.k, self.v, self.n + nq, self.scale, o, self.lse_self)
        if advance:
            self.n += nq
        return o

    def step_cross(self, q, out=None):
        o = self.o_cross if out is None else out
        L.fastar_dense_attn(q, self.kp, self.vp, self.P, self.scale, o, self.lse_cross)
        return o

    def step(self, q, k_cur, v_cur, advance: bool = True, timer=None):
        nq = q.shape[1]
        main = torch.cuda.current_stream()
        t = timer or (lambda *a: None)
        L.fastar_dense_append(k_cur, v_cur, self.k, self.v, self.n)
        nk = self.n + nq
        t("dense_attn", main, "begin")
        L.fastar_dense_attn(q, self.k, self.v, nk, self.scale, self.o_self, self.lse_self)
        t("dense_attn", main, "end")
        L.fastar_dense_attn(q, self.kp, self.vp, self.P, self.scale, self.o_cross, self.lse_cross)
        if advance:
            self.n = nk
        return self.o_self, self.o_cross
