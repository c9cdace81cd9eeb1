"""CPU oracle of OTIL's selective latent transmit (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use
this module.  Plain numpy, fp64 for the scores; it shares no code with the CUDA path.

Source: "OTIL for SDXL on 4x L40S".
  * "What is implemented where", Vectorised selection: each step every rank scores the
    K sub-blocks of its own slice, sends the top k (one topk, one index_select) and every
    receiver writes them into its copy with one index_copy_ per peer.
  * Same section: the dynamic-polling rule "unvisited blocks first, then the highest
    dissimilarity" is topk(dissimilarity + 10 * unvisited, k), cosine dissimilarity lying
    in [0, 2]; the selection covers every sub-block within ceil(K / k) steps.
  * "Self-tests": the local slice is bit-exact fresh, a remote position is either a
    received sub-block or stale memory and never a blend, exactly k blocks arrive from
    each peer, and finalize() gives every rank the exact latent.
  * "Read this before interpreting the numbers", item 3: the transmitted tensor is the
    noise prediction at latent resolution, [B, C, H, W] = 2 x 4 x 128 x 128.

Readings where the page is silent (each listed with its reason in the design notes):
rank p owns rows [p*H/P, (p+1)*H/P) (the row patches of the method); a sub-block is a
bh x bw spatial tile of that band over every batch and channel, numbered row-major over
the band; the dissimilarity of a sub-block is 1 - cos(fresh, peers' copy), with cos = 0
when either norm is 0; ties in the score go to the lower sub-block index; the
unvisited flags are cleared by a synchronous step (finalize with reset) and nowhere else;
the peers' copy of band p is the same on every receiver, so any receiver's copy serves.
"""
from __future__ import annotations

import numpy as np

UNVISITED_BONUS = 10.0  # above any dissimilarity (cosine dissimilarity <= 2)


def sub_blocks(H: int, W: int, P: int, bh: int, bw: int):
    """(row0, col0) of each sub-block of a band, relative to the band, row-major."""
    Hp = H // P
    return [(r, c) for r in range(0, Hp, bh) for c in range(0, W, bw)]


def block_view(t: np.ndarray, p: int, i: int, P: int, bh: int, bw: int):
    """The [B, C, bh, bw] slice of sub-block i of band p of a [B, C, H, W] tensor."""
    B, C, H, W = t.shape
    r, c = sub_blocks(H, W, P, bh, bw)[i]
    r0 = p * (H // P) + r
    return t[:, :, r0:r0 + bh, c:c + bw]


def dissimilarity(x: np.ndarray, s: np.ndarray) -> float:
    """1 - cos(x, s) in fp64; cos = 0 when either vector is zero."""
    x = np.asarray(x, np.float64).ravel()
    s = np.asarray(s, np.float64).ravel()
    nx, ns = np.sqrt(np.dot(x, x)), np.sqrt(np.dot(s, s))
    if nx == 0.0 or ns == 0.0:
        return 1.0
    return 1.0 - float(np.dot(x, s)) / (nx * ns)


def scores(fresh: np.ndarray, views: np.ndarray, visited: np.ndarray, P: int, bh: int, bw: int):
    """[P, K] selection scores: dissimilarity of each sub-block against the peers' copy,
    plus UNVISITED_BONUS for sub-blocks not sent since the last reset."""
    B, C, H, W = fresh.shape
    K = len(sub_blocks(H, W, P, bh, bw))
    out = np.zeros((P, K))
    for p in range(P):
        peer = (p + 1) % P
        for i in range(K):
            d = dissimilarity(block_view(fresh, p, i, P, bh, bw),
                              block_view(views[peer], p, i, P, bh, bw))
            out[p, i] = d + (0.0 if visited[p, i] else UNVISITED_BONUS)
    return out


def select_top_k(score_row: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k highest scores, ties to the lower index, in ascending order."""
    order = sorted(range(len(score_row)), key=lambda i: (-score_row[i], i))
    return np.array(sorted(order[:k]), dtype=np.int64)


def apply_selection(fresh: np.ndarray, views: np.ndarray, visited: np.ndarray, sel: np.ndarray,
                    P: int, bh: int, bw: int):
    """One exchange with the given selection [P, k]: returns (views, visited, messages).

    Rank p's message is its k selected fresh sub-blocks (index_select); every other rank
    copies them into its copy of band p (index_copy_); rank p's own band becomes its
    fresh band in full.  Copies only: no value is ever blended.
    """
    views = np.array(views, copy=True)
    visited = np.array(visited, copy=True)
    B, C, H, W = fresh.shape
    Hp = H // P
    k = sel.shape[1]
    msg = np.zeros((P, k, B, C, bh, bw), dtype=fresh.dtype)
    for p in range(P):
        for j, i in enumerate(sel[p]):
            msg[p, j] = block_view(fresh, p, int(i), P, bh, bw)
            visited[p, int(i)] = 1
            for r in range(P):
                if r != p:
                    block_view(views[r], p, int(i), P, bh, bw)[...] = msg[p, j]
        views[p][:, :, p * Hp:(p + 1) * Hp] = fresh[:, :, p * Hp:(p + 1) * Hp]
    return views, visited, msg


def exchange_step(fresh, views, visited, P: int, bh: int, bw: int, k: int):
    """Score, select and apply (the whole step); returns (views, visited, sel, msg)."""
    sc = scores(fresh, views, visited, P, bh, bw)
    sel = np.stack([select_top_k(sc[p], k) for p in range(P)])
    views, visited, msg = apply_selection(fresh, views, visited, sel, P, bh, bw)
    return views, visited, sel, msg


def finalize(fresh, views, visited, reset: bool):
    """The exact gather: every rank's view becomes the fresh latent; with reset (the
    synchronous step) the unvisited flags are set again."""
    views = np.broadcast_to(fresh, views.shape).copy()
    visited = np.zeros_like(visited) if reset else np.array(visited, copy=True)
    return views, visited
