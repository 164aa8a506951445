"""The bench's algorithmic-byte accounting of attention launches (host logic,
no GPU): the library's trace counts K/V bytes for B sequences of the longest
context, and the bench rescales them to the keys each sequence reads."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_equal_contexts_keep_the_trace_count():
    assert bench.attention_key_ratio([2048], 17, 2048) == 1.0
    assert bench.attention_key_ratio([4096] * 4, 17, 4096) == 1.0


def test_ragged_contexts_count_each_sequence_once():
    # keys read: (100 + 17) + (500 + 17); counted by the trace: 2 * (500 + 17)
    assert bench.attention_key_ratio([100, 500], 17, 500) == (117 + 517) / (2 * 517)


def test_ragged_batch_16_workload_ratio_matches_its_drawn_lengths():
    wl = synth.WORKLOADS["qwen3_8b_L5_ragged_B16"]
    lens = synth.ctx_lengths(wl)
    r = bench.attention_key_ratio(lens, wl.rows, int(lens.max()))
    per_seq = sum(int(n) + wl.rows for n in lens)
    assert np.isclose(r, per_seq / (wl.batch * (int(lens.max()) + wl.rows)))
    assert 0.5 < r < 0.7   # contexts U{512..8192}: mean well below the longest
