"""Shared-memory bank model of the 128-key-tile prefill's rel boxes.

Each softmax warp of prefill_wide_kernel reads its 32 rows (4 apart: row
4 lane + q4) from the four 32-row rel boxes of a tile slot, 17 8-byte loads
per lane.  The boxes are kRelColsW bf16 distances wide, and the odd boxes
start kRelOddShift distances lower.  This model recomputes every lane's
address as scores_with_bias_w2 forms it, for every lane quarter q4, every
alignment of the tile's first row and both column halves.  It checks that
each load stays inside its box row and costs two wavefronts, the least for
256 bytes; the unshifted 168-wide layout it replaced costs four.

The constants are read from csrc/relattn_prefill.cuh, so a change there is
checked here on the CPU.
"""

import os
import re
from collections import defaultdict

HERE = os.path.dirname(os.path.abspath(__file__))
HDR = os.path.join(os.path.dirname(HERE), "paged_relative_bias_gb300", "csrc",
                   "relattn_prefill.cuh")


def constant(name):
    src = open(HDR).read()
    m = re.search(r"\b%s = (\d+)[;,]" % name, src)
    assert m, name
    return int(m.group(1))


def worst_wavefronts(cols, shift, box_rows):
    """Largest number of distinct 32-bit words one bank serves for one 8-byte
    load of a warp, over every case the kernel meets."""
    worst = 0
    box_elems = box_rows * cols
    for q4 in range(4):
        for align in range(8):  # (P0 + 1) & 7
            for half in range(2):
                for k in range(17):
                    words = defaultdict(set)
                    for lane in range(32):
                        r = 4 * lane + q4
                        rbox, rrow = r // box_rows, r % box_rows
                        col = rrow + align + 64 * (1 - half) + shift * (rbox & 1)
                        # the 17 loads of 4 distances stay inside the row
                        assert (col & ~3) + 68 <= cols, (col, cols)
                        elem = rbox * box_elems + rrow * cols + (col & ~3) + 4 * k
                        w = elem // 2  # bf16 -> 32-bit word
                        for ww in (w, w + 1):
                            words[ww % 32].add(ww)
                    worst = max(worst, max(len(v) for v in words.values()))
    return worst


def test_rel_box_reads_take_two_wavefronts():
    cols = constant("kRelColsW")
    shift = constant("kRelOddShift")
    rows = constant("kRelBoxRows")
    assert worst_wavefronts(cols, shift, rows) == 2


def test_unshifted_narrow_boxes_would_conflict():
    # the layout the odd-box shift replaced: 168 distances, no shift
    assert worst_wavefronts(168, 0, constant("kRelBoxRows")) == 4


def test_box_rows_and_slot_size():
    cols = constant("kRelColsW")
    rows = constant("kRelBoxRows")
    src = open(HDR).read()
    assert "kRelBoxBytesW = kRelBoxRows * kRelColsW * 2" in src
    box_bytes = rows * cols * 2
    # each box starts on a 128-byte boundary (a tensor copy's destination)
    assert box_bytes % 128 == 0
    # a row needs 128 distances, 32 rows 159, plus up to 7 for rounding the
    # start down to 16 bytes and the odd boxes' shift
    assert cols >= 128 + 31 + 7 + constant("kRelOddShift")
