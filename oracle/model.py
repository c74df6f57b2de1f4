"""The Llama-architecture decode step, prefill and KV fork, plain fp64.

Weights come as the quantised bytes the library also receives (a dict with
``tok_embd``, ``output`` (None when tied to the embedding), ``output_norm``
and a per-layer list of dicts with ``attn_norm``, ``ffn_norm``, ``wq``,
``wk``, ``wv``, ``wo``, ``w_gate``, ``w_up``, ``w_down``).  Matrices are
[out x in] with Q8_0 / Q4_0 blocks along ``in``.

Per token at position pos (the engine page, section 1 and section 4.4; the
SwarmKV page, section 2: decode reads the per-layer KV cache filled by
prefill and extends it by one token):

    x  = dequant(tok_embd[token])
    for each layer:
        xn = rmsnorm(x, attn_norm)
        q, k, v = Wq xn, Wk xn, Wv xn
        q, k = rope(q, pos), rope(k, pos)
        K[pos], V[pos] = fp16(k), fp16(v)          # the cache is fp16
        o  = attention(q, K[0..pos], V[0..pos])    # causal, GQA
        x  = x + Wo o
        xn = rmsnorm(x, ffn_norm)
        x  = x + Wdown (silu(Wgate xn) * (Wup xn))
    logits = Wout rmsnorm(x, output_norm)          # Wout = tok_embd when tied

Prefill runs the same math for T tokens at positions 0..T-1 at once and
returns the last token's logits (reading: the pages do not say which logits
prefill yields; the last token's are the ones decoding continues from).

The fork (SwarmKV page, sections 3-4) copies the source sequence's cache; a
branch then continues at positions prefix_len, prefix_len + 1, ...

Layer skip and self-speculative decoding (the engine page, sections 2.5,
3.5, 4.5 and 5.3): a decode step may skip layers (their output is their
input); the speculative loop drafts with skipped layers and keeps only the
tokens the full model would pick.
"""
from __future__ import annotations

import numpy as np

from . import kquant, ops, quant


class OracleSeq:
    """One sequence's fp16-valued K/V cache, per layer, held in fp64."""

    def __init__(self, n_layers: int, n_kv_heads: int, head_dim: int, capacity: int = 64):
        self.n_layers, self.nkv, self.hd = n_layers, n_kv_heads, head_dim
        self.k = [np.zeros((capacity, n_kv_heads, head_dim)) for _ in range(n_layers)]
        self.v = [np.zeros((capacity, n_kv_heads, head_dim)) for _ in range(n_layers)]
        self.lens = [0] * n_layers
        self.n = 0   # positions consumed; a layer skipped at a step appends nothing there

    @property
    def length(self) -> int:
        return self.n

    def _reserve(self, layer: int, n: int):
        cap = self.k[layer].shape[0]
        if n > cap:
            new = max(n, 2 * cap)
            for arr in (self.k, self.v):
                grown = np.zeros((new, self.nkv, self.hd))
                grown[:cap] = arr[layer]
                arr[layer] = grown

    def append(self, layer: int, pos0: int, k: np.ndarray, v: np.ndarray):
        """Store fp16-rounded k, v [T, nkv, hd] at positions pos0..pos0+T-1."""
        if pos0 != self.lens[layer]:
            raise ValueError(f"layer {layer}: append at {pos0} but cache holds {self.lens[layer]}")
        T = k.shape[0]
        self._reserve(layer, pos0 + T)
        self.k[layer][pos0:pos0 + T] = ops.round_f16(k)
        self.v[layer][pos0:pos0 + T] = ops.round_f16(v)
        self.lens[layer] = pos0 + T
        self.n = max(self.n, pos0 + T)

    def truncate(self, n: int):
        """Forget positions >= n in every layer (the sequence continues at n)."""
        if not 0 <= n <= self.n:
            raise ValueError(f"truncate to {n} of a sequence of length {self.n}")
        self.lens = [min(v, n) for v in self.lens]
        self.n = n

    def keys(self, layer: int) -> np.ndarray:
        return self.k[layer][: self.lens[layer]]

    def values(self, layer: int) -> np.ndarray:
        return self.v[layer][: self.lens[layer]]

    def fork(self) -> "OracleSeq":
        """A copy of the cache: the branch starts where the prefix ended."""
        c = OracleSeq(self.n_layers, self.nkv, self.hd, 1)
        c.k = [a.copy() for a in self.k]
        c.v = [a.copy() for a in self.v]
        c.lens = list(self.lens)
        c.n = self.n
        return c

    def set_layer(self, layer: int, k: np.ndarray, v: np.ndarray):
        """Load a layer's cache from given fp16-valued arrays [n, nkv, hd]."""
        n = k.shape[0]
        self._reserve(layer, n)
        self.k[layer][:n] = k
        self.v[layer][:n] = v
        self.lens[layer] = n
        self.n = max(self.n, n)


class OracleModel:
    """fp64 forward of a quantised Llama-architecture model.

    ``cfg`` needs: n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn,
    vocab, rope_theta, rms_eps, wtype, tied.  Dequantised matrices are cached
    up to ``cache_bytes``; larger models dequantise rows in chunks per call.

    Every matrix is in the format ``cfg.wtype`` (8: Q8_0, 4: Q4_0) unless
    ``weights["formats"]`` maps its (layer, name) to another: "q4_k", "q5_k"
    or "q6_k" (a K-quant file mixes these per matrix, Q4_K_M for instance;
    layer None for tok_embd and output).
    """

    def __init__(self, cfg, weights: dict, cache_bytes: int = 2 << 30, chunk_rows: int = 8192):
        self.cfg = cfg
        self.w = weights
        self.cache_bytes = cache_bytes
        self.chunk_rows = chunk_rows
        self._cache: dict = {}
        self._cached = 0
        H, hd = cfg.hidden, cfg.head_dim
        self.shapes = {
            "wq": (cfg.n_heads * hd, H), "wk": (cfg.n_kv_heads * hd, H), "wv": (cfg.n_kv_heads * hd, H),
            "wo": (H, cfg.n_heads * hd), "w_gate": (cfg.ffn, H), "w_up": (cfg.ffn, H),
            "w_down": (H, cfg.ffn), "tok_embd": (cfg.vocab, H), "output": (cfg.vocab, H),
        }

    # -- weights -------------------------------------------------------------

    def _blocks(self, layer, name):
        if layer is None:
            if name == "output" and self.w.get("output") is None:
                return self.w["tok_embd"]
            return self.w[name]
        lw = self.w["layers"][layer]
        if lw is None:
            raise ValueError(f"layer {layer} weights were not generated")
        return lw[name]

    def _rows(self, layer, name, r0: int, r1: int) -> np.ndarray:
        """Rows [r0, r1) of one matrix, dequantised from its own format."""
        cols = self.shapes[name][1]
        if name == "output" and layer is None and self.w.get("output") is None:
            name = "tok_embd"
        fmt = self.w.get("formats", {}).get((layer, name), self.cfg.wtype)
        blocks = self._blocks(layer, name)
        if fmt in (8, 4):
            return quant.matrix_rows(blocks, cols, fmt, r0, r1)
        return kquant.matrix_rows(blocks, cols, fmt, r0, r1)

    def matrix(self, layer, name) -> np.ndarray:
        """Dequantised fp64 [rows, cols] of one matrix (cached when it fits)."""
        key = (layer, name)
        if key in self._cache:
            return self._cache[key]
        rows, cols = self.shapes[name]
        m = self._rows(layer, name, 0, rows)
        if self._cached + m.nbytes <= self.cache_bytes:
            self._cache[key] = m
            self._cached += m.nbytes
        return m

    def matmul(self, layer, name, x: np.ndarray, rows=None) -> np.ndarray:
        """y = W x for x [cols] or [T, cols]; optionally only selected output rows."""
        nrows, cols = self.shapes[name]
        key = (layer, name)
        if rows is not None:
            out = []
            for r in np.asarray(rows).ravel():
                w = self._rows(layer, name, int(r), int(r) + 1)
                out.append(x @ w[0])
            return np.stack(out, axis=-1)
        if key in self._cache or nrows * cols * 8 <= self.cache_bytes - self._cached:
            return x @ self.matrix(layer, name).T
        parts = []
        for r0 in range(0, nrows, self.chunk_rows):
            r1 = min(nrows, r0 + self.chunk_rows)
            w = self._rows(layer, name, r0, r1)
            parts.append(x @ w.T)
        return np.concatenate(parts, axis=-1)

    def norm_gain(self, layer, name) -> np.ndarray:
        if layer is None:
            return np.asarray(self.w["output_norm"], dtype=np.float64)
        return np.asarray(self.w["layers"][layer][name], dtype=np.float64)

    # -- the step --------------------------------------------------------------

    def new_seq(self, capacity: int = 64) -> OracleSeq:
        return OracleSeq(self.cfg.n_layers, self.cfg.n_kv_heads, self.cfg.head_dim, capacity)

    def embed(self, tokens) -> np.ndarray:
        """Dequantised embedding rows: [T, hidden] (or [hidden] for one id)."""
        toks = np.atleast_1d(np.asarray(tokens))
        rows = [self._rows(None, "tok_embd", int(t), int(t) + 1)[0] for t in toks]
        x = np.stack(rows)
        return x if np.ndim(tokens) else x[0]

    def layer_forward(self, layer: int, x: np.ndarray, pos0: int, seq: OracleSeq) -> np.ndarray:
        """One layer for T tokens at positions pos0..pos0+T-1; extends seq's cache."""
        cfg = self.cfg
        single = x.ndim == 1
        X = np.atleast_2d(x)
        T = X.shape[0]
        nh, nkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        xn = ops.rmsnorm(X, self.norm_gain(layer, "attn_norm"), cfg.rms_eps)
        q = self.matmul(layer, "wq", xn).reshape(T, nh, hd)
        k = self.matmul(layer, "wk", xn).reshape(T, nkv, hd)
        v = self.matmul(layer, "wv", xn).reshape(T, nkv, hd)
        pos = pos0 + np.arange(T)
        q = ops.rope(q, pos, cfg.rope_theta)
        k = ops.rope(k, pos, cfg.rope_theta)
        seq.append(layer, pos0, k, v)
        if single:
            o = ops.attention(q[0], seq.keys(layer), seq.values(layer))[None]
        else:
            o = ops.causal_attention(q, seq.keys(layer), seq.values(layer), q_pos0=pos0)
        X = X + self.matmul(layer, "wo", o.reshape(T, nh * hd))
        xn = ops.rmsnorm(X, self.norm_gain(layer, "ffn_norm"), cfg.rms_eps)
        h = ops.swiglu(self.matmul(layer, "w_gate", xn), self.matmul(layer, "w_up", xn))
        X = X + self.matmul(layer, "w_down", h)
        return X[0] if single else X

    def final_logits(self, x: np.ndarray, rows=None) -> np.ndarray:
        """Final RMSNorm and LM head (optionally only the given vocab rows)."""
        xn = ops.rmsnorm(x, self.norm_gain(None, "output_norm"), self.cfg.rms_eps)
        return self.matmul(None, "output", xn, rows=rows)

    def decode_step(self, seq: OracleSeq, token: int, pos: int, capture: list | None = None,
                    skip=()) -> np.ndarray:
        """Logits [vocab] for `token` at position `pos` (= the cache length).

        ``skip``: layers not computed at this step (the engine page, sections
        2.5 / 3.5 / 4.5: a skipped layer's output is the previous layer's
        output); they append nothing to their cache.
        """
        if pos != seq.length:
            raise ValueError(f"pos {pos} != sequence length {seq.length}")
        x = self.embed(int(token))
        for l in range(self.cfg.n_layers):
            if l not in skip:
                x = self.layer_forward(l, x, pos, seq)
            if capture is not None:
                capture.append(x.copy())
        seq.n = pos + 1
        return self.final_logits(x)

    def layer_cosines(self, seq: OracleSeq, token: int, pos: int) -> np.ndarray:
        """One decode step of `token` at `pos`; for every layer, the cosine
        similarity of its output with its input (the previous layer's output,
        the embedding row for layer 0): the calibration the engine page
        describes for layer skipping (sections 3.5 and 4.5: layers whose
        output is more than 0.98 similar to the previous one are skipped)."""
        x0 = self.embed(int(token))
        cap = []
        self.decode_step(seq, token, pos, capture=cap)
        ins = [x0] + cap[:-1]
        return np.array([ops.cosine(a, b) for a, b in zip(ins, cap)])

    def prefill(self, seq: OracleSeq, tokens, capture: list | None = None,
                all_logits: bool = False) -> np.ndarray:
        """All prompt tokens through every layer at once, at positions
        length .. length+T-1; the last token's logits, or every token's
        ([T, vocab]) with all_logits."""
        toks = np.asarray(tokens)
        pos0 = seq.length
        X = self.embed(toks)
        for l in range(self.cfg.n_layers):
            X = self.layer_forward(l, X, pos0, seq)
            if capture is not None:
                capture.append(X[-1].copy())
        seq.n = pos0 + len(toks)
        return self.final_logits(X) if all_logits else self.final_logits(X[-1])

    def greedy_decode(self, seq: OracleSeq, token: int, n_steps: int, skip=()):
        """n_steps greedy steps from `token` at the sequence end; (tokens, logits)."""
        toks, logits = [], []
        for _ in range(n_steps):
            lg = self.decode_step(seq, token, seq.length, skip=skip)
            logits.append(lg)
            token = ops.greedy(lg)
            toks.append(token)
        return toks, logits

    def speculative_decode(self, seq: OracleSeq, token: int, n_tokens: int, draft_skip, k: int):
        """Greedy self-speculative decoding (the engine page, sections 3.5 and
        5.3: a cheap draft proposes tokens, the full model checks them in one
        pass).  The draft is this model with the layers in ``draft_skip``
        skipped.  Each round, with the current token t at position P:

          1. the draft decodes r = min(k, tokens still wanted - 1) greedy
             tokens d_1..d_r from t (its layers fill the cache at P..P+r-1);
          2. the sequence is cut back to P and the full model runs
             [t, d_1, .., d_r] at positions P..P+r at once (a prefill that
             keeps every row's logits), giving greedy tokens v_0..v_r;
          3. the longest prefix with d_i == v_{i-1} is accepted (n tokens);
             the round emits d_1..d_n and v_n, and the sequence keeps
             positions up to P+n (t, d_1..d_n), continuing with v_n.

        Returns (tokens [n_tokens], stats {rounds, drafted, accepted,
        min_gap}).  The tokens are the full model's greedy continuation: a
        draft token is kept only where the full model picks it too.  min_gap
        is the smallest top-2 logit gap of any greedy pick made (draft or
        full), i.e. how far the run is from a tie.
        """
        out = []
        stats = {"rounds": 0, "drafted": 0, "accepted": 0, "min_gap": np.inf}
        cur = int(token)
        skip = set(draft_skip)
        while len(out) < n_tokens:
            P = seq.length
            r = min(k, n_tokens - len(out) - 1)
            drafts = []
            t = cur
            for i in range(r):
                lg = self.decode_step(seq, t, P + i, skip=skip)
                stats["min_gap"] = min(stats["min_gap"], ops.top2_gap(lg))
                t = ops.greedy(lg)
                drafts.append(t)
            seq.truncate(P)
            rows = self.prefill(seq, [cur] + drafts, all_logits=True)
            stats["min_gap"] = min([stats["min_gap"]] + [ops.top2_gap(lg) for lg in rows])
            v = [ops.greedy(lg) for lg in rows]
            n = 0
            while n < r and drafts[n] == v[n]:
                n += 1
            out += drafts[:n] + [v[n]]
            seq.truncate(P + n + 1)
            cur = v[n]
            stats["rounds"] += 1
            stats["drafted"] += r
            stats["accepted"] += n
        return out, stats
