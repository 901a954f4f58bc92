"""Shard ownership, causal visibility and tile classes, by plain enumeration.

TEST INFRASTRUCTURE (see oracle/__init__.py): never imported by the product path.

The ring cuts the token axis into P shards of S = N / P tokens:
  * contiguous: shard u holds tokens [u*S, (u+1)*S) ("Part 4: Ring Attention"
    (Fofadiya) 4.3.1 "Initial State"; "Ring Attention: what the near-infinite
    context paper actually says", "The ring mechanism, step by step": device 0
    holds tokens 0 .. N/P-1, device 1 the next N/P, ...).
  * striped: token t belongs to shard t mod P at local index t div P ("Ring
    Attention" (aarnphm.xyz): Striped Attention keeps the ring schedule but
    alternates shard ownership).  N must be divisible by P ("...near-infinite
    context paper...", "Production tradeoffs": devices must divide the
    sequence length evenly).
  * zigzag: the sequence is cut into 2P chunks of C = N / 2P tokens and shard u
    holds chunk u (local 0 .. C-1) then chunk 2P-1-u (local C .. 2C-1)
    ("Part 4: Ring Attention" 4.8.3 "Zigzag (Striped) Load Balancing"; Transformer
    Math "Ring Attention" (aicassindra), "Causal masking wastes half the ring").
    N must be divisible by 2P.
The causal mask is defined on global positions: key position <= query position
("...near-infinite context paper...", "The causal masking complication";
Transformer Math "Ring Attention" (aicassindra), "Composing with tensor
parallelism": positions are global).  A shard pair / tile with no admitted
(query, key) pair can be skipped ("Part 4" 4.8.1 "Skipping Fully-Masked Blocks").
"""
from __future__ import annotations

from typing import List, Tuple

CONTIGUOUS = "contiguous"
STRIPED = "striped"
ZIGZAG = "zigzag"
LAYOUTS = (CONTIGUOUS, STRIPED, ZIGZAG)

TILE_EMPTY = 0      # no admitted pair: skipped
TILE_PARTIAL = 1    # some pairs admitted: needs an element mask
TILE_FULL = 2       # every pair admitted: no mask


def _check(layout: str, N: int, P: int) -> int:
    if layout not in LAYOUTS:
        raise ValueError(f"unknown layout {layout!r}")
    if N <= 0 or P <= 0 or N % P != 0:
        raise ValueError("N and P must be positive with N divisible by P")
    if layout == ZIGZAG and N % (2 * P) != 0:
        raise ValueError("zigzag needs N divisible by 2P")
    return N // P


def owner(layout: str, N: int, P: int, t: int) -> int:
    """Shard that holds global token t."""
    S = _check(layout, N, P)
    if layout == ZIGZAG:
        c = t // (S // 2)                  # chunk of the token
        return c if c < P else 2 * P - 1 - c
    return t // S if layout == CONTIGUOUS else t % P


def local_index(layout: str, N: int, P: int, t: int) -> int:
    """Position of token t inside its shard."""
    S = _check(layout, N, P)
    if layout == ZIGZAG:
        C = S // 2
        c = t // C
        return t % C if c < P else C + t % C
    return t % S if layout == CONTIGUOUS else t // P


def token_of(layout: str, N: int, P: int, u: int, i: int) -> int:
    """Global token (= global position) of local index i in shard u."""
    S = _check(layout, N, P)
    if layout == ZIGZAG:
        C = S // 2
        return u * C + i if i < C else (2 * P - 1 - u) * C + (i - C)
    return u * S + i if layout == CONTIGUOUS else i * P + u


def shard_map(layout: str, N: int, P: int) -> Tuple[List[int], List[int], List[int]]:
    """(owner[t], local[t]) for every token t, and token_of[u*S + i]."""
    S = _check(layout, N, P)
    own = [owner(layout, N, P, t) for t in range(N)]
    loc = [local_index(layout, N, P, t) for t in range(N)]
    tok = [token_of(layout, N, P, u, i) for u in range(P) for i in range(S)]
    return own, loc, tok


def shard_tokens(layout: str, N: int, P: int, u: int) -> List[int]:
    """Global tokens of shard u in local order."""
    S = _check(layout, N, P)
    return [token_of(layout, N, P, u, i) for i in range(S)]


def visible(layout: str, N: int, P: int, causal: bool, u: int, i: int, b: int, j: int) -> bool:
    """Whether local query i of shard u may attend to local key j of shard b."""
    if not causal:
        return True
    return token_of(layout, N, P, b, j) <= token_of(layout, N, P, u, i)


def mask_block(layout: str, N: int, P: int, causal: bool, u: int, b: int) -> List[List[bool]]:
    """Element mask [S][S] for queries of shard u against keys of shard b."""
    S = _check(layout, N, P)
    return [[visible(layout, N, P, causal, u, i, b, j) for j in range(S)] for i in range(S)]


def tile_class(layout: str, N: int, P: int, causal: bool, u: int, b: int,
               i0: int, j0: int, tile_m: int, tile_n: int) -> int:
    """Class of the tile rows [i0, i0+tile_m) x keys [j0, j0+tile_n) of the
    (u, b) shard pair, counting only in-range rows and keys (< S), found by
    enumerating every pair."""
    S = _check(layout, N, P)
    n_in = n_ok = 0
    for i in range(i0, min(i0 + tile_m, S)):
        for j in range(j0, min(j0 + tile_n, S)):
            n_in += 1
            n_ok += visible(layout, N, P, causal, u, i, b, j)
    if n_ok == 0:
        return TILE_EMPTY
    return TILE_FULL if n_ok == n_in else TILE_PARTIAL


def tile_classes(layout: str, N: int, P: int, causal: bool, u: int, b: int,
                 tile_m: int, tile_n: int) -> List[List[int]]:
    """All tile classes of the (u, b) pair, [ceil(S/tile_m)][ceil(S/tile_n)]."""
    S = _check(layout, N, P)
    return [[tile_class(layout, N, P, causal, u, b, i0, j0, tile_m, tile_n)
             for j0 in range(0, S, tile_n)] for i0 in range(0, S, tile_m)]


def nonempty_shard_pairs(layout: str, N: int, P: int, causal: bool) -> int:
    """How many (u, b) shard pairs admit at least one (query, key) pair."""
    S = _check(layout, N, P)
    cnt = 0
    for u in range(P):
        for b in range(P):
            if any(visible(layout, N, P, causal, u, i, b, j)
                   for i in range(S) for j in range(S)):
                cnt += 1
    return cnt
