"""bench.py's launch count (the `gpu_launches` claim) follows kv_rotate_qk's documented
dispatch: one kernel below 128 x 152 dense (row, head) pairs, else the tensor-core kernel plus
one for the exact copies / Hadamard rows when there are any; then one flush and one decode."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_decode_sized_steps_launch_three_kernels():
    for w in (synth.TINY_GQA4, synth.QWEN3_8B_32K, synth.QWEN3_4B_B64, synth.QWEN3_32B_128K):
        assert bench.step_launches(w, w.batch, w.batch * w.n_new, w.ring_cap) == 3


def test_chunk_step_launches_four_kernels():
    w = synth.WUSH_CHUNK_B16                       # dense keys on the tensor cores, copied values
    assert bench.rotate_launches(w, w.batch, w.batch * w.n_new) == 2
    assert bench.step_launches(w, w.batch, w.batch * w.n_new, w.ring_cap) == 4


def test_rotate_dispatch_edges():
    w = synth.WUSH_CHUNK_B16
    rows = bench.TC_MIN_PAIRS // w.n_kv_heads
    assert bench.rotate_launches(w, 0, rows - 1) == 1               # just below the threshold
    assert bench.rotate_launches(w, 0, rows) == 2
    dense_v = w.replace(value_transform="orthogonal")
    assert bench.rotate_launches(dense_v, 0, rows) == 1               # no copies left over
    had = synth.QWEN3_32B_128K.replace(value_transform="orthogonal")
    assert bench.rotate_launches(had, 0, rows) == 2                   # Hadamard rows + dense V
    assert bench.rotate_launches(w, 0, 0) == 0
