"""Accepted-path KV compaction, plain numpy (test infrastructure only).

Source: EAGLE-2 page, §"一段更贴近实现的流程", the step after verification: the accepted tokens
and their KV are committed to the cache and the rejected candidates' temporary KV is discarded;
§"工程实现里的几个难点": the tree's KV lives in a temporary area while it is verified.

Readings taken where the page is silent:

* The verify forward computes one temporary KV row per tree position, position 0 being the root
  (the token committed last round, whose KV is not yet in the cache). A round therefore commits
  accept_len + 1 rows: the root and the accepted path's positions, in path order. The bonus
  token's KV is computed by the next round's forward (it is the next root).
* A KV row is an opaque byte string of fixed length (all layers, keys and values, of one token).
* The cache of request b holds cache_len[b] committed rows; the new rows go to positions
  cache_len[b], cache_len[b] + 1, ...; a round that would pass the cache's capacity is an error
  and commits nothing for that request.
"""

import numpy as np


def commit_kv(tmp_kv, cache, cache_len, accept_len, accept_path, row_off=None):
    """Append the root's and the accepted positions' KV rows to each request's cache (in place).

    tmp_kv [B][P][row], cache [B][L_max][row] (any dtype), cache_len [B] (updated), accept_len [B],
    accept_path [B][D_path] (positions, root first, -1 padded). With ``row_off`` ([B+1], the
    padding-free layout of ``oracle.tree.packed_row_offsets``) tmp_kv is [rows][row] and position i
    of request b is its row row_off[b] + i. Returns the list of requests whose commit was refused
    for lack of room.
    """
    B, L_max = cache.shape[0], cache.shape[1]

    def tmp_row(b, i):
        return tmp_kv[int(row_off[b]) + i] if row_off is not None else tmp_kv[b, i]

    refused = []
    for b in range(B):
        n = int(accept_len[b]) + 1
        start = int(cache_len[b])
        if start + n > L_max:
            refused.append(b)
            continue
        for j in range(n):
            cache[b, start + j] = tmp_row(b, int(accept_path[b, j]))
        cache_len[b] = start + n
    return refused
