"""Masked softmax attention over an explicit token-level chunk mask -- oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Everything here is
float64 on the given (already bf16-rounded) inputs, uses one library matmul
per product and otherwise follows the definitions below line by line.

Definitions and their sources
-----------------------------
Block-causal chunk visibility -- "WanToFight: Real-Time Generative Game Engine
for Multi-Player Combat Interaction", section 三 (技术架构), table "模型组件",
row "Block-Causal Attention", and section "训练流程 / Stage 2 (因果适配)": inside a
chunk attention is bidirectional; across chunks a query sees its own chunk and
the 2 chunks before it, never a later chunk.  With a general window W:

    query token in chunk qc sees key token in chunk kc  iff  0 <= qc - kc <= W

"WorldPlay2: Extending Real-Time Interactive World Models in Control and
Horizon", Figure 3 (causal attention mask for compressed memory training) and
"Matrix-Game 4.0: Harnessing Video Models for Real-Time Playable Game Worlds",
section "前置知识 / 因果自回归与 KV 缓存" (recent window plus a reference frame)
add a permanent prefix, the sink / reference chunk, that every query sees.

Attention on the visible set (the textbook scaled-dot-product definition):

    s_ij  = scale * sum_d q_id k_jd
    P_ij  = exp(s_ij) / sum_{j' visible} exp(s_ij')        (j visible)
    O_i   = sum_j P_ij v_j
    LSE_i = ln sum_{j visible} exp(s_ij)                    (natural log)

Log-sum-exp merge of a key partition -- "Matrix-Game 4.0", sections
"前置知识 / 因果自回归与 KV 缓存" and "技术新颖性": the KV window is cut into
intervals computed in parallel and their partial outputs are merged with
log-sum-exp.  For parts s with (O_s, L_s) computed on disjoint key subsets:

    L = ln sum_s exp(L_s),    O = sum_s exp(L_s - L) O_s

(an empty part has L_s = -inf and weight 0).

Readings where the pages are silent: LSE is the natural log of the scaled
scores; a query row with no visible key (never produced by a valid call) gives
O = 0 and LSE = -inf.
"""

from __future__ import annotations

import numpy as np

from .ring import ListRing, RingError

SINK_CHUNK = -(10**9)  # chunk id given to sink tokens in the explicit mask


def chunk_visibility(q_chunk: np.ndarray, k_chunk: np.ndarray, window: int,
                     k_is_sink: np.ndarray | None = None) -> np.ndarray:
    """Explicit token-level mask ``[Lq, Nk]`` from per-token chunk ids."""
    qc = np.asarray(q_chunk, dtype=np.int64)[:, None]
    kc = np.asarray(k_chunk, dtype=np.int64)[None, :]
    d = qc - kc
    mask = (d >= 0) & (d <= int(window))
    if k_is_sink is not None:
        mask = mask | np.asarray(k_is_sink, dtype=bool)[None, :]
    return mask


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray,
                     scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Attention of one head: q ``[Lq, D]``, k ``[Nk, D]``, v ``[Nk, Dv]``,
    mask bool ``[Lq, Nk]``.  Returns (O ``[Lq, Dv]``, LSE ``[Lq]``) in float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    mask = np.asarray(mask, dtype=bool)
    s = float(scale) * (q @ k.T)
    s = np.where(mask, s, -np.inf)
    any_visible = mask.any(axis=1)
    m = np.where(any_visible, np.max(s, axis=1), 0.0)
    e = np.where(mask, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    safe_l = np.where(any_visible, l, 1.0)
    p = e / safe_l[:, None]
    o = p @ v
    o = np.where(any_visible[:, None], o, 0.0)
    lse = np.where(any_visible, m + np.log(safe_l), -np.inf)
    return o, lse


def lse_merge(parts_o, parts_lse) -> tuple[np.ndarray, np.ndarray]:
    """Merge partial results over a partition of the keys.

    ``parts_o``: sequence of ``[..., Dv]`` arrays, ``parts_lse``: matching
    ``[...]`` arrays (``-inf`` for an empty part)."""
    lses = np.stack([np.asarray(x, dtype=np.float64) for x in parts_lse])
    os_ = np.stack([np.asarray(x, dtype=np.float64) for x in parts_o])
    big_m = np.max(lses, axis=0)
    finite = np.isfinite(big_m)
    mm = np.where(finite, big_m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - mm[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(finite, mm + np.log(np.where(finite, tot, 1.0)), -np.inf)
    coef = np.where(np.isfinite(lses), np.exp(lses - np.where(finite, lse, 0.0)[None]), 0.0)
    o = (coef[..., None] * os_).sum(axis=0)
    return o, lse


def streaming_key_set(ring: ListRing, chunk: int, k_cur, v_cur, window: int, use_sink: bool):
    """Keys visible to the queries of ``chunk`` in streaming inference.

    Candidates are the sink (if used), every chunk held in the list ring that
    is not later than ``chunk`` (earlier than ``chunk`` when ``k_cur`` is
    given) and, when given, the freshly computed current chunk ``k_cur``.
    Visibility is then decided by the explicit token mask.  Raises
    ``RingError`` when a chunk the window needs is not held.

    ``k_cur`` / ``v_cur`` and the ring records are ``[B, H, Lc, D]``; returns
    K, V ``[B, H, Nk, D]``, per-token chunk ids ``[Nk]`` and sink flags.
    """
    chunk = int(chunk)
    ks, vs, ids, sink_flags = [], [], [], []
    if use_sink:
        if ring.sink is None:
            raise RingError("sink requested but not set")
        sk, sv = ring.sink
        n = sk.shape[2]
        ks.append(sk); vs.append(sv); ids.append(np.full(n, SINK_CHUNK)); sink_flags.append(np.ones(n, bool))
    held = set()
    for c, k, v in ring.records:
        if c > chunk or (k_cur is not None and c == chunk):
            continue
        held.add(c)
        n = k.shape[2]
        ks.append(k); vs.append(v); ids.append(np.full(n, c)); sink_flags.append(np.zeros(n, bool))
    if k_cur is not None:
        held.add(chunk)
        n = np.asarray(k_cur).shape[2]
        ks.append(np.asarray(k_cur)); vs.append(np.asarray(v_cur))
        ids.append(np.full(n, chunk)); sink_flags.append(np.zeros(n, bool))
    for c in range(max(0, chunk - int(window)), chunk + 1):
        if c not in held:
            raise RingError(f"chunk {c} needed by the window of chunk {chunk} is not held")
    return (np.concatenate(ks, axis=2), np.concatenate(vs, axis=2),
            np.concatenate(ids), np.concatenate(sink_flags))


def streaming_chunk_attention(q_bhld, ring: ListRing, chunk: int, k_cur, v_cur, window: int,
                              use_sink: bool, scale: float):
    """Streaming chunk attention for one chunk's queries ``[B, H, Lq, D]``.

    Returns (O ``[B, H, Lq, D]``, LSE ``[B, H, Lq]``) in float64."""
    q = np.asarray(q_bhld, dtype=np.float64)
    K, V, kid, ksink = streaming_key_set(ring, chunk, k_cur, v_cur, window, use_sink)
    B, H, Lq, _ = q.shape
    mask = chunk_visibility(np.full(Lq, int(chunk)), kid, window, ksink)
    O = np.empty(q.shape[:3] + (V.shape[3],), dtype=np.float64)
    L = np.empty((B, H, Lq), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = masked_attention(q[b, h], K[b, h], V[b, h], mask, scale)
    return O, L


def block_causal_attention(q_blhd, k_blhd, v_blhd, chunk_tokens: int, window: int, scale: float,
                           rows=None, heads=None, batches=None, restrict_keys: bool = True):
    """Block-causal attention over a whole sequence (training shape).

    Inputs are token-major ``[B, L, H, D]``; token t belongs to chunk
    ``t // chunk_tokens``.  ``rows`` (query token indices), ``heads`` and
    ``batches`` select which outputs to evaluate (default: all); each query
    row is computed independently from the definition with the explicit mask.
    Returns (O ``[nb, nh, nrows, D]``, LSE ``[nb, nh, nrows]``).

    The selected rows are taken one query chunk qc at a time.  With
    ``restrict_keys`` the candidate keys of that group are the tokens of
    chunks max(0, qc - W) .. qc: every other key is masked for every row of
    the group, so its term of the definition is an exact zero and leaving it
    out changes no sum (only the order in which zeros would be added).  The
    explicit mask is still applied to the candidates.  ``restrict_keys=False``
    scores every row against all L keys.
    """
    q = np.asarray(q_blhd)
    k = np.asarray(k_blhd)
    v = np.asarray(v_blhd)
    B, L, H, _ = q.shape
    Lc = int(chunk_tokens)
    rows = np.arange(L) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = range(H) if heads is None else list(heads)
    batches = range(B) if batches is None else list(batches)
    key_chunk = np.arange(L) // Lc
    O = np.empty((len(batches), len(heads), len(rows), v.shape[3]), dtype=np.float64)
    LSE = np.empty((len(batches), len(heads), len(rows)), dtype=np.float64)
    q_chunk = rows // Lc
    groups = []  # (positions in `rows`, candidate key slice)
    for qc in np.unique(q_chunk):
        pos = np.nonzero(q_chunk == qc)[0]
        kr = slice(max(0, int(qc) - int(window)) * Lc, min(L, (int(qc) + 1) * Lc)) if restrict_keys else slice(0, L)
        step = 2048  # rows per matmul (memory bound only)
        for p0 in range(0, len(pos), step):
            groups.append((pos[p0:p0 + step], kr))
    for bi, b in enumerate(batches):
        for hi, h in enumerate(heads):
            kk = np.asarray(k[b, :, h, :], dtype=np.float64)
            vv = np.asarray(v[b, :, h, :], dtype=np.float64)
            for pos, kr in groups:
                rr = rows[pos]
                mask = chunk_visibility(rr // Lc, key_chunk[kr], window)
                o, lse = masked_attention(np.asarray(q[b, rr, h, :], dtype=np.float64), kk[kr], vv[kr], mask, scale)
                O[bi, hi, pos] = o
                LSE[bi, hi, pos] = lse
    return O, LSE
