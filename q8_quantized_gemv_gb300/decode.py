"""The per-token projection sequence of a synthetic decoder, run through the
C ABI.  Two dataflows:

glu=True (a pre-norm decoder layer):
    x = norm(h) -> q, k, v;  quantize(o_in) -> o;
    h' = h + o, x = norm(h') -> gate/up -> SwiGLU -> quantize -> down;
    h'' = h' + down, x = norm(h'') -> next layer (the last: the lm-head norm)
  the residual add, norm and quantizer run as one launch
  (lk_add_rmsnorm_quant) and the SwiGLU with its quantizer runs in the
  gate/up launch's epilogue (lk_gemv_q8_glu);
glu=False (the default: the projections alone):
    norm -> quantize -> q, k, v; quantize -> o; norm -> quantize -> fused
    gate/up; quantize -> down; the o output feeds the MLP norm and the down
    output the next layer's norm, with no residual add.
Then RMSNorm -> quantize -> lm-head with the argmax epilogue -> argmax.

Attention is not part of the projection path, so the input it would produce
for the o projection is a fixed seeded vector (N(0,1) with 1% x20 outliers,
one per layer) quantized every token; with glu=False the down projection's
input is such a vector too.

Weights live on the device for the life of the object (about 8 GB for the
36-layer, hidden-4096 configuration); every buffer is allocated once here and
``run_token`` only launches kernels, so it can be captured in a CUDA graph.
"""
from __future__ import annotations

import torch

from . import lk, synth


class DecodeStack:
    def __init__(self, layers=36, hidden=4096, q_dim=4096, kv_dim=1024, ffn=12288, vocab=151936,
                 batch=1, mode=lk.LK_INT8ACT, seed=synth.SEED_BASE + 4, device="cuda", eps=1e-6,
                 fused=False, chain=False, group_qkv=True, prefill=None, glu=False, fused_qkv=True, pdl=False,
                 path=0, tune=None, splitk=True):
        self.L, self.H, self.Q, self.KV, self.F, self.V = layers, hidden, q_dim, kv_dim, ffn, vocab
        self.B, self.mode, self.eps, self.dev = batch, lk._mode(mode), eps, torch.device(device)
        # per projection (qkv, o, gu, down, lm): warps of a GEMV block that
        # fill their stages before the dependency wait (lk_launch_cfg.prefill)
        self.prefill = dict(prefill or {})
        # every launch a programmatic dependent of the one before (may be
        # changed between tokens); the GEMV kernel (lk_launch_cfg.path)
        self.pdl = bool(pdl)
        self.path = lk.PATHS[path] if isinstance(path, str) else int(path)
        # further lk_launch_cfg fields for every call (tensor-core layouts ...)
        self.tune = dict(tune or {})
        dev = self.dev
        s = seed
        # the gated pair runs as one fused launch; the chain and fused-prologue
        # forms keep the projections-alone dataflow
        self.glu = bool(glu) and not chain and not fused
        self.shapes = {"q": (q_dim, hidden), "k": (kv_dim, hidden), "v": (kv_dim, hidden),
                       "o": (hidden, q_dim), "gu": (2 * ffn, hidden), "down": (hidden, ffn)}
        # fused_qkv: q, k and v are row ranges of one [q + 2 kv, hidden]
        # matrix (the usual fused attention projection); the per-launch
        # sequence then runs them as ONE GEMV over its rows
        self.fused_qkv = bool(fused_qkv)
        self.layers = []
        for l in range(layers):
            w = {}
            if self.fused_qkv:
                w["qkv"] = synth.q8_matrix_torch(q_dim + 2 * kv_dim, hidden, s + 1000 * l + 30, dev)
                bounds = {"q": (0, q_dim), "k": (q_dim, q_dim + kv_dim), "v": (q_dim + kv_dim, q_dim + 2 * kv_dim)}
                for n, (r0, r1) in bounds.items():
                    w[n] = (w["qkv"][0][r0:r1], w["qkv"][1][r0:r1])
            for i, (name, (N, K)) in enumerate(self.shapes.items()):
                if name in ("q", "k", "v") and self.fused_qkv:
                    continue
                if name == "gu" and self.glu:
                    # the gate and up matrices of the pair (ffn rows each)
                    w["gate"] = synth.q8_matrix_torch(ffn, hidden, s + 1000 * l + i, dev)
                    w["up"] = synth.q8_matrix_torch(ffn, hidden, s + 1000 * l + 20 + i, dev)
                    continue
                w[name] = synth.q8_matrix_torch(N, K, s + 1000 * l + i, dev)
            w["g_attn"] = synth.norm_gain_torch(hidden, s + 1000 * l + 10, dev)
            w["g_mlp"] = synth.norm_gain_torch(hidden, s + 1000 * l + 11, dev)
            w["o_in"] = synth.activation_torch(batch, q_dim, s + 1000 * l + 12, dev, outliers=True)
            w["d_in"] = synth.activation_torch(batch, ffn, s + 1000 * l + 13, dev, outliers=True)
            self.layers.append(w)
        self.lm = synth.q8_matrix_torch(vocab, hidden, s + 999_000, dev)
        self.g_final = synth.norm_gain_torch(hidden, s + 999_001, dev)
        self.x0 = synth.activation_torch(batch, hidden, s + 999_002, dev, outliers=True)

        f32, i8 = torch.float32, torch.int8
        B = batch
        self.h = torch.empty((B, hidden), dtype=f32, device=dev)        # residual stream
        self.xn = torch.empty((B, hidden), dtype=f32, device=dev)       # normed (Dequant GEMV input)
        self.acts = {K: self._act_bufs(K) for K in {hidden, q_dim, ffn}}
        self.out = {name: torch.empty((B, N), dtype=f32, device=dev) for name, (N, _) in self.shapes.items()}
        if self.fused_qkv:
            # one output for the fused matrix; q, k, v are its column ranges
            self.out_qkv = torch.empty((B, q_dim + 2 * kv_dim), dtype=f32, device=dev)
            self.qkv_views = {"q": self.out_qkv[:, :q_dim], "k": self.out_qkv[:, q_dim:q_dim + kv_dim],
                              "v": self.out_qkv[:, q_dim + kv_dim:]}
        if self.glu:
            self.hbuf = [torch.empty((B, hidden), dtype=f32, device=dev) for _ in range(2)]  # residual stream
            self.gu_buf = torch.empty((2, B, ffn), dtype=f32, device=dev)   # gate and up values
            self.hglu = torch.empty((B, ffn), dtype=f32, device=dev)        # SwiGLU output (Dequant input)
            self.glu_cnt = torch.zeros((ffn // 32,), dtype=torch.int32, device=dev)
        self.logits = torch.empty((B, vocab), dtype=f32, device=dev)
        self.parts = torch.zeros((B * lk.lk_argmax_parts_max(vocab),), dtype=torch.int64, device=dev)
        self.idx = torch.empty((B,), dtype=torch.int32, device=dev)
        self.n_parts = 0
        # one launch per projection (norm/quantize prologue inside the ring
        # GEMV) wherever the ring kernel takes the shape and lk_gemv_q8 would
        # not pick the tensor-core kernel (2..8 rows); else norm/quantize
        # kernels followed by lk_gemv_q8
        shapes = dict(self.shapes, lm=(vocab, hidden))
        self.kernel = {n: lk.lk_gemv_kernel_for(N, K, self.mode, B, 0, cfg=self._cfg())
                       for n, (N, K) in shapes.items()}
        ring_cfg = lk.launch_cfg(path=2)
        ring = {n: lk.lk_gemv_kernel_for(N, K, self.mode, B, 0, cfg=ring_cfg) == 2 for n, (N, K) in shapes.items()}
        # fused: True / False for every projection, or the names of those
        # that compute their own norm/quantize prologue
        want = set(shapes) if fused is True else set() if not fused else set(fused)
        self.fused = {n: n in want and ring[n] and self.kernel[n] != 3 for n in shapes}
        # the whole token as one cooperative chain launch (the ring kernel's
        # fused steps), where every step fits
        self.x_buf = self.x0.clone()  # the token's input rows
        self.chain = None
        if chain and all(ring.values()):
            self.chain = lk.Chain(self._chain_ops(), dev)
        # q, k and v of a layer as one grouped launch (a chain without
        # barriers: one prologue, the three weight streams back to back)
        self.qkv = None
        if self.chain is None and group_qkv and all(self.fused[n] for n in ("q", "k", "v")) and not self.fused_qkv:
            self.qkv = []
            for l, w in enumerate(self.layers):
                x = self.x_buf if l == 0 else self.h
                self.qkv.append(lk.Chain([lk.chain_op(w[n][0], w[n][1], x, self.out[n], gain=w["g_attn"])
                                          for n in ("q", "k", "v")], dev))

        fq = [self.fused[n] for n in ("q", "k", "v")]
        self.qkv_one = self.fused_qkv and self.chain is None and (all(fq) or not any(fq))
        if self.qkv_one:
            self.out.update(self.qkv_views)
        # split-K at 2 or more activation rows (the tensor-core kernel holds a
        # chunk of the activation per block, so long rows keep more weight
        # stages in flight): the chunk count the library favours for each
        # projection (lk_splitk_chunks_for; 1 = the plain GEMV).  splitk=False
        # turns it off, a dict {projection: S} sets it.
        cand = {}
        if self.qkv_one and not any(fq):
            cand["qkv"] = (q_dim + 2 * kv_dim, hidden)
        for n in ("o", "gu", "down"):
            if not self.fused[n] and not (n == "gu" and self.glu):
                cand[n] = self.shapes[n]
        if splitk is False or B < 2 or self.chain is not None:
            self.splitk = {}
        elif isinstance(splitk, dict):
            self.splitk = {n: int(v) for n, v in splitk.items() if n in cand and int(v) > 1}
        else:
            self.splitk = {n: S for n, (N, K) in cand.items() if (S := lk.lk_splitk_chunks_for(N, K, self.mode, B)) > 1}
        self.part = {n: torch.empty((S * B * cand[n][0],), dtype=f32, device=dev) for n, S in self.splitk.items()}

    def _act_bufs(self, K):
        B = self.B
        d = {"xq": torch.empty((B, K), dtype=torch.int8, device=self.dev),
             "xs": torch.empty((B, K // 32), dtype=torch.float32, device=self.dev)}
        if self.mode == lk.LK_TWOPASS:
            d["xl"] = torch.empty((B, K), dtype=torch.int8, device=self.dev)
        return d

    # -- the launches of one token ---------------------------------------------------
    def _norm(self, x, g):
        """RMSNorm -> quantize; returns the GEMV activation arguments."""
        if self.mode == lk.LK_DEQUANT:
            lk.lk_rmsnorm_quant(x, g, self.mode, self.eps, self.xn, cfg=self._cfg())
            return {"x": self.xn}
        a = self.acts[x.shape[1]]
        lk.lk_rmsnorm_quant(x, g, self.mode, self.eps, None, a["xq"], a.get("xl"), a["xs"], cfg=self._cfg())
        return a

    def _add_norm(self, x, r, s, g):
        """s = x + r, then RMSNorm -> quantize of s (one launch); returns the
        GEMV activation arguments."""
        if self.mode == lk.LK_DEQUANT:
            lk.lk_add_rmsnorm_quant(x, r, g, self.mode, self.eps, s=s, xn=self.xn, cfg=self._cfg())
            return {"x": self.xn}
        a = self.acts[x.shape[1]]
        lk.lk_add_rmsnorm_quant(x, r, g, self.mode, self.eps, s=s, xq=a["xq"], xl=a.get("xl"), xs=a["xs"],
                                cfg=self._cfg())
        return a

    def _quant(self, x):
        if self.mode == lk.LK_DEQUANT:
            return {"x": x}
        a = self.acts[x.shape[1]]
        lk.lk_quantize_act(x, self.mode, a["xq"], a.get("xl"), a["xs"], cfg=self._cfg())
        return a

    def _cfg(self, name=None):
        """Launch settings of one call: pdl and the GEMV kernel of the stack,
        and for projection `name` the warps filling before the dependency
        wait, where set."""
        return lk.launch_cfg(**dict(self.tune, pdl=self.pdl, path=self.path,
                                    prefill=self.prefill.get(name, 0) if name else 0))

    def _gemv(self, w, y, acts, parts=None, name=None):
        S = self.splitk.get(name, 1)
        if S > 1 and parts is None:
            # the split-K partials, then their combine in ascending chunk order
            c = self._cfg(name)
            lk.lk_gemv_q8_splitk(w[0], w[1], self.mode, S, self.part[name], M=self.B, cfg=c, **acts)
            lk.lk_splitk_combine(self.mode, self.part[name], S, self.B, w[0].shape[0], y, cfg=c)
            return 0
        return lk.lk_gemv_q8(w[0], w[1], self.mode, y, M=self.B, argmax_parts=parts, cfg=self._cfg(name), **acts)

    def _chain_ops(self):
        """The token's steps.  A step waits (grid barrier) where a decoder's
        dataflow has a dependency: the attention output before o, o before
        gate/up, the gated activation before down, down before the next
        layer's q/k/v and the lm-head -- including where the synthetic o and
        down inputs would not need it."""
        ops = []
        x = self.x_buf
        for l, w in enumerate(self.layers):
            for name in ("q", "k", "v"):
                ops.append(lk.chain_op(w[name][0], w[name][1], x, self.out[name], gain=w["g_attn"],
                                       wait=(name == "q" and l > 0)))
            ops.append(lk.chain_op(w["o"][0], w["o"][1], w["o_in"], self.out["o"], wait=True))
            ops.append(lk.chain_op(w["gu"][0], w["gu"][1], self.out["o"], self.out["gu"], gain=w["g_mlp"],
                                   wait=True))
            ops.append(lk.chain_op(w["down"][0], w["down"][1], w["d_in"], self.h, wait=True))
            x = self.h
        ops.append(lk.chain_op(self.lm[0], self.lm[1], x, self.logits, gain=self.g_final,
                               argmax_parts=self.parts, argmax_idx=self.idx, wait=True))
        return ops

    def _qkv_launch(self, w, a):
        """The attention projections of layer weights w on activation a: one
        GEMV over the fused q|k|v matrix, or one grouped GEMV over three."""
        c = self._cfg("qkv")
        if self.fused_qkv:
            return lambda: self._gemv(w["qkv"], self.out_qkv, a, name="qkv")
        return lambda: lk.lk_gemv_q8_group([(w[n][0], w[n][1], self.out[n]) for n in ("q", "k", "v")], self.mode,
                                           M=self.B, cfg=c, **a)

    def _run_token_glu(self, hook):
        """The pre-norm decoder layer dataflow (glu=True)."""
        def launch(name, fn):
            return fn() if hook is None else hook(name, fn)

        m, B, L = self.mode, self.B, self.L
        a_h = self._norm(self.x_buf, self.layers[0]["g_attn"])
        h_cur = self.x_buf
        for l, w in enumerate(self.layers):
            launch("qkv", self._qkv_launch(w, a_h))
            a_o = self._quant(w["o_in"])
            launch("o", lambda w=w, a=a_o: self._gemv(w["o"], self.out["o"], a, name="o"))
            h_mid = self.hbuf[0]
            a_m = self._add_norm(self.out["o"], h_cur, h_mid, w["g_mlp"])
            a_d = {"x": self.hglu} if m == lk.LK_DEQUANT else self.acts[self.F]
            launch("gu", lambda w=w, a=a_m, d=a_d: lk.lk_gemv_q8_glu(
                w["gate"][0], w["gate"][1], w["up"][0], w["up"][1], m, self.gu_buf, h=self.hglu,
                hq=d.get("xq"), hl=d.get("xl"), hs=d.get("xs"), cnt=self.glu_cnt, M=B, cfg=self._cfg("gu"), **a))
            launch("down", lambda w=w, d=a_d: self._gemv(w["down"], self.out["down"], d, name="down"))
            h_next = self.hbuf[1]
            g_next = self.layers[l + 1]["g_attn"] if l + 1 < L else self.g_final
            a_h = self._add_norm(self.out["down"], h_mid, h_next, g_next)
            h_cur = h_next
        self.n_parts = launch("lm", lambda: self._gemv(self.lm, self.logits, a_h, self.parts, name="lm"))
        lk.lk_argmax(self.idx, B, self.V, parts=self.parts, n_parts=self.n_parts)
        return self.idx

    def run_token(self, x_in=None, hook=None):
        """Launch one token's sequence on the current stream and return the
        device int32 [B] argmax.  ``hook``, if given, is called as
        hook(name, launch) around each GEMV launch (for per-kernel timing)."""
        if x_in is not None and x_in.data_ptr() != self.x_buf.data_ptr():
            self.x_buf.copy_(x_in)
        if self.glu:
            return self._run_token_glu(hook)
        if self.chain is not None and hook is None:
            lk.lk_gemv_chain(self.chain, self.mode, self.B, self.eps, cfg=self._cfg())
            return self.idx

        def g(name, w, y, x, gain, parts=None, acts=None):
            """Launch one projection; returns (launch result, the activation
            arguments it used when not fused)."""
            if self.fused[name]:
                def launch():
                    return lk.lk_rmsnorm_quant_gemv_q8(w[0], w[1], self.mode, x, y, gain=gain, eps=self.eps,
                                                       argmax_parts=parts, cfg=self._cfg(name))
                a = None
            else:
                a = acts if acts is not None else (self._norm(x, gain) if gain is not None else self._quant(x))

                def launch():
                    return self._gemv(w, y, a, parts, name)
            return (launch() if hook is None else hook(name, launch)), a

        x = self.x_buf
        for l, w in enumerate(self.layers):
            if self.qkv is not None:
                def launch(c=self.qkv[l]):
                    return lk.lk_gemv_chain(c, self.mode, self.B, self.eps, cfg=self._cfg("qkv"))
                launch() if hook is None else hook("qkv", launch)
            elif self.qkv_one and self.fused["q"]:
                # one launch: norm -> quantize prologue, the fused q|k|v matrix
                def launch(w=w, x=x):
                    return lk.lk_rmsnorm_quant_gemv_q8(w["qkv"][0], w["qkv"][1], self.mode, x, self.out_qkv,
                                                       gain=w["g_attn"], eps=self.eps, cfg=self._cfg("qkv"))
                launch() if hook is None else hook("qkv", launch)
            elif not any(self.fused[n] for n in ("q", "k", "v")):
                # one norm, then q, k and v as one GEMV over the fused matrix
                # (or one grouped GEMV over the three)
                a = self._norm(x, w["g_attn"])
                launch = self._qkv_launch(w, a)
                launch() if hook is None else hook("qkv", launch)
            else:
                # q, k and v read the same normed activation: quantized once
                _, a = g("q", w["q"], self.out["q"], x, w["g_attn"])
                g("k", w["k"], self.out["k"], x, w["g_attn"], acts=a if not self.fused["k"] else None)
                g("v", w["v"], self.out["v"], x, w["g_attn"], acts=a if not self.fused["v"] else None)
            g("o", w["o"], self.out["o"], w["o_in"], None)
            g("gu", w["gu"], self.out["gu"], self.out["o"], w["g_mlp"])
            g("down", w["down"], self.h, w["d_in"], None)
            x = self.h
        self.n_parts, _ = g("lm", self.lm, self.logits, x, self.g_final, self.parts)
        lk.lk_argmax(self.idx, self.B, self.V, parts=self.parts, n_parts=self.n_parts)
        return self.idx

    # -- accounting ------------------------------------------------------------------------
    def weight_bytes(self, name=None):
        """Algorithmic weight bytes (N*K levels + N*K/16 scale bytes)."""
        def mb(N, K):
            return N * K + N * K // 16
        if name == "lm":
            return mb(self.V, self.H)
        if name is not None:
            return mb(*self.shapes[name])  # "gu": the gate/up pair together
        return self.L * sum(mb(N, K) for N, K in self.shapes.values()) + mb(self.V, self.H)

    def glu_launches(self):
        """Launches of the gate/up pair: one (the ring kernel's SwiGLU
        epilogue) at one activation row where the ring kernel takes the
        shape, else the grouped GEMVs and the SwiGLU kernel."""
        ring = lk.lk_gemv_kernel_for(2 * self.F, self.H, self.mode, 1, 0, cfg=lk.launch_cfg(path=2)) == 2
        return 1 if (self.B == 1 and ring and self.path == 0) else 2

    def launches_per_token(self):
        if self.chain is not None:
            return 1
        if self.glu:
            # first norm; per layer q/k/v, [quantize], o, add+norm, gate/up
            # pair, down, add+norm (and a combine per split-K projection);
            # lm-head, argmax
            per_layer = 5 + (0 if self.mode == lk.LK_DEQUANT else 1) + self.glu_launches() + len(self.splitk)
            return 1 + self.L * per_layer + 2
        n = 1  # argmax reduce
        f = self.fused
        qkv_norm = 0 if (f["q"] and f["k"] and f["v"]) else 1  # one shared norm for q, k, v
        # q, k, v in one launch: the fused chain, or lk_gemv_q8_group on the
        # tensor-core or chain kernel (both take the shape where the ring does)
        grouped = self.qkv is not None or self.qkv_one or \
            (not any(f[n] for n in ("q", "k", "v")) and self.kernel["q"] in (2, 3))
        per_layer = (4 if grouped else 6) + qkv_norm \
            + (0 if (f["o"] or self.mode == lk.LK_DEQUANT) else 1) + (0 if f["gu"] else 1) \
            + (0 if (f["down"] or self.mode == lk.LK_DEQUANT) else 1) + len(self.splitk)
        return n + self.L * per_layer + 1 + (0 if f["lm"] else 1)


class BlkDecodeStack:
    """The projections-alone decode sequence with every matrix in one of the
    other GGUF block formats (lk_gemv_blk): per layer RMSNorm -> q|k|v (one
    fused matrix) -> quantize -> o -> RMSNorm -> gate/up -> quantize -> down;
    then RMSNorm -> lm-head -> argmax of the logits.  One to LK_MAX_M
    activation rows, every mode; synthetic weights of the format's layout
    (synth.blk_matrix), the same activations and gains as DecodeStack."""

    def __init__(self, fmt, layers=36, hidden=4096, q_dim=4096, kv_dim=1024, ffn=12288, vocab=151936, batch=1,
                 mode=lk.LK_INT8ACT, seed=synth.SEED_BASE + 4, device="cuda", eps=1e-6, pdl=True):
        self.fmt = fmt
        self.L, self.H, self.Q, self.KV, self.F, self.V = layers, hidden, q_dim, kv_dim, ffn, vocab
        self.B, self.mode, self.eps, self.dev = batch, lk._mode(mode), eps, torch.device(device)
        self.pdl = bool(pdl)
        dev, s = self.dev, seed
        self.shapes = {"qkv": (q_dim + 2 * kv_dim, hidden), "o": (hidden, q_dim), "gu": (2 * ffn, hidden),
                       "down": (hidden, ffn)}
        self.layers = []
        for l in range(layers):
            w = {n: synth.blk_matrix_torch(fmt, N, K, s + 1000 * l + i, dev)
                 for i, (n, (N, K)) in enumerate(self.shapes.items())}
            w["g_attn"] = synth.norm_gain_torch(hidden, s + 1000 * l + 10, dev)
            w["g_mlp"] = synth.norm_gain_torch(hidden, s + 1000 * l + 11, dev)
            w["o_in"] = synth.activation_torch(batch, q_dim, s + 1000 * l + 12, dev, outliers=True)
            w["d_in"] = synth.activation_torch(batch, ffn, s + 1000 * l + 13, dev, outliers=True)
            self.layers.append(w)
        self.lm = synth.blk_matrix_torch(fmt, vocab, hidden, s + 999_000, dev)
        self.g_final = synth.norm_gain_torch(hidden, s + 999_001, dev)
        self.x0 = synth.activation_torch(batch, hidden, s + 999_002, dev, outliers=True)
        self.x_buf = self.x0.clone()
        f32, B = torch.float32, batch
        self.h = torch.empty((B, hidden), dtype=f32, device=dev)
        self.xn = {K: torch.empty((B, K), dtype=f32, device=dev) for K in {hidden, q_dim, ffn}}
        self.acts = {}
        for K in {hidden, q_dim, ffn}:
            d = {"xq": torch.empty((B, K), dtype=torch.int8, device=dev),
                 "xs": torch.empty((B, K // 32), dtype=torch.float32, device=dev)}
            if self.mode == lk.LK_TWOPASS:
                d["xl"] = torch.empty((B, K), dtype=torch.int8, device=dev)
            self.acts[K] = d
        self.out = {n: torch.empty((B, N), dtype=f32, device=dev) for n, (N, _) in self.shapes.items()}
        self.logits = torch.empty((B, vocab), dtype=f32, device=dev)
        self.scratch = torch.zeros((B * lk.lk_argmax_scratch_entries(vocab),), dtype=torch.int64, device=dev)
        self.idx = torch.empty((B,), dtype=torch.int32, device=dev)

    def _cfg(self):
        return lk.launch_cfg(pdl=1 if self.pdl else 0)

    def _norm(self, x, g):
        K = x.shape[1]
        if self.mode == lk.LK_DEQUANT:
            lk.lk_rmsnorm_quant(x, g, self.mode, self.eps, self.xn[K], cfg=self._cfg())
            return {"x": self.xn[K]}
        a = self.acts[K]
        lk.lk_rmsnorm_quant(x, g, self.mode, self.eps, None, a["xq"], a.get("xl"), a["xs"], cfg=self._cfg())
        return a

    def _quant(self, x):
        if self.mode == lk.LK_DEQUANT:
            return {"x": x}
        a = self.acts[x.shape[1]]
        lk.lk_quantize_act(x, self.mode, a["xq"], a.get("xl"), a["xs"], cfg=self._cfg())
        return a

    def _gemv(self, w, K, y, a):
        lk.lk_gemv_blk(self.fmt, w, K, self.mode, y, M=self.B, cfg=self._cfg(), **a)

    def run_token(self, x_in=None, hook=None):
        """One token on the current stream; returns the device int32 [B]
        argmax.  ``hook(name, launch)``, if given, wraps each GEMV launch."""
        if x_in is not None and x_in.data_ptr() != self.x_buf.data_ptr():
            self.x_buf.copy_(x_in)

        def g(name, w, K, y, a):
            def launch():
                return self._gemv(w, K, y, a)
            return launch() if hook is None else hook(name, launch)

        x = self.x_buf
        for w in self.layers:
            g("qkv", w["qkv"], self.H, self.out["qkv"], self._norm(x, w["g_attn"]))
            g("o", w["o"], self.Q, self.out["o"], self._quant(w["o_in"]))
            g("gu", w["gu"], self.H, self.out["gu"], self._norm(self.out["o"], w["g_mlp"]))
            g("down", w["down"], self.F, self.h, self._quant(w["d_in"]))
            x = self.h
        g("lm", self.lm, self.H, self.logits, self._norm(x, self.g_final))
        lk.lk_argmax(self.idx, self.B, self.V, logits=self.logits, scratch=self.scratch)
        return self.idx

    def weight_bytes(self, name=None):
        """The format's bytes of one token's matrices (or of projection `name`)."""
        def mb(N, K):
            return N * lk.lk_format_row_bytes(self.fmt, K)
        if name == "lm":
            return mb(self.V, self.H)
        if name is not None:
            return mb(*self.shapes[name])
        return self.L * sum(mb(N, K) for N, K in self.shapes.values()) + mb(self.V, self.H)

    def launches_per_token(self):
        quant = 0 if self.mode == lk.LK_DEQUANT else 2
        return self.L * (6 + quant) + 3
