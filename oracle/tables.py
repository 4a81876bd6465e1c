"""Brute-force enumeration of the varlen chunk tables.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Chunks of `chunk` tokens restart at every document start; the last chunk of a
document holds the remaining len mod chunk tokens (or a full chunk).  The
flashinfer Cake GDN pages keep four chunk tables and a segment table built
from cu_seqlens ("feat(cake_gdn_kcp) ... #8172" page, commit note on the
backend's fifth table); their contents are not printed, so the tables here are
this library's own definition:

  chunk_offsets[N+1]  index of each document's first chunk (prefix sum)
  chunk_doc[NC]       document of each chunk
  chunk_tok0[NC]      first token (global) of each chunk
  chunk_len[NC]       number of tokens in each chunk (1..chunk)
"""
from __future__ import annotations

import numpy as np


def chunk_tables(cu_seqlens, chunk=64):
    cu = [int(x) for x in cu_seqlens]
    offsets, doc, tok0, clen = [0], [], [], []
    for d in range(len(cu) - 1):
        t = cu[d]
        while t < cu[d + 1]:
            doc.append(d)
            tok0.append(t)
            clen.append(min(chunk, cu[d + 1] - t))
            t += chunk
        offsets.append(len(doc))
    as32 = lambda x: np.array(x, dtype=np.int32)
    return dict(chunk_offsets=as32(offsets), chunk_doc=as32(doc), chunk_tok0=as32(tok0),
                chunk_len=as32(clen))
