"""In-place paged prefill relabels a prefill chunk's rows as paged decode
rows (synth.prefill_as_decode). On the oracle, both readings of the same
chunk must give the same results: this pins the relabelling on the CPU."""

import numpy as np
import pytest

import oracle
from sparse_attention_top_expand_gb300 import synth


def test_paged_rows_give_the_gathered_rows_results():
    inp = synth.prefill_chunk(seed=21, seq_lens=(700, 1100), queries_per_seq=6, num_heads=16,
                              page_size=32, cbs=64, ncb=5, topk=100)
    kv, ks = oracle.gather_reference(inp)
    dec = synth.prefill_as_decode(inp)
    assert dec.rows == inp.rows
    rows = list(range(inp.rows))
    a = oracle.reference_rows(inp, rows=rows, mode="dense", contig=(kv, ks))
    b = oracle.reference_rows(dec, rows=rows, mode="dense")
    for r in rows:
        assert a[r].end == b[r].end
        assert np.array_equal(a[r].sparse_indices, b[r].sparse_indices)
        assert np.array_equal(a[r].topk, b[r].topk)
        assert np.array_equal(a[r].logits, b[r].logits, equal_nan=True)


def test_rows_must_start_at_their_sequence():
    inp = synth.prefill_chunk(seed=21, seq_lens=(700, 1100), queries_per_seq=6, num_heads=16,
                              page_size=32, cbs=64, ncb=5, topk=100)
    inp.cu_seqlen_ks = inp.cu_seqlen_ks.copy()
    inp.cu_seqlen_ks[3] += 1
    with pytest.raises(ValueError):
        synth.prefill_as_decode(inp)
