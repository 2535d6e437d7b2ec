"""Held-out shared-load patterns for the oracle's wide-access bank model.

The oracle's rule for 64- and 128-bit shared loads (oracle/oracle_f64.c,
oracle_shared_request) was fitted to the ncu wavefront counts of the 26 lane
patterns in lds_wavefronts_sm103.txt.  The patterns below were chosen
afterwards and not used for that fit: new permutations, strided and
broadcast mixes, and the exact lane offsets of the product kernels' own
fragment reads.  Their measured counts are in lds_wavefronts_heldout_sm103.txt,
and tests/test_bank_model.py checks that the unchanged model predicts them.

Run on a GPU, this script launches smem_bank_pattern_probe once per pattern
(each lane's word offsets are what the probe reads, shifted by whole bank
rows between accesses),
in the order of PATTERNS, so that

    ncu --clock-control none -k regex:bank_pattern_kernel \\
        --metrics l1tex__data_pipe_lsu_wavefronts_mem_shared_op_ld.sum,smsp__inst_executed_op_shared_ld.sum \\
        --csv python tests/golden/lds_heldout_patterns.py

gives the wavefronts per load instruction of each pattern (launch i is
pattern i).  It holds no bank arithmetic; the expected values come from the
measurement.
"""
import os
import sys

# (width in bytes, name, lane -> index of the width-sized chunk); chunk c
# starts at word c * width / 4
EXPRS = [
    "lane ^ 1",
    "31 - lane",
    "(lane * 3) & 31",
    "(lane * 5) & 63",
    "(lane & 7) * 2",
    "(lane >> 2) * 3",
    "lane % 3",
    "(lane >> 1) * 2",
    "16 * (lane & 1)",
    "8 * (lane & 3) + (lane >> 3)",
    "(lane * 9) & 63",
    "(lane >> 3) + 4 * (lane & 1)",
]
# the product kernels' fragment reads, as the library reports them
# (sgemm_f32_smem_request kind, warp, step, stage)
KERNEL_READS = [
    (2, 5, 7, 1, "8 x 8 kernels, A fragment read"),
    (3, 6, 20, 2, "8 x 8 kernels, B fragment read"),
    (11, 2, 9, 2, "k-major 8 x 16 kernels, A fragment read"),
    (12, 3, 37, 1, "k-major 8 x 16 kernels, B fragment read"),
]
WIDE = [(w, e) for e in EXPRS for w in (16, 8)]
NARROW = [(4, "(lane * 33) & 63"), (4, "(lane >> 1) * 32"), (4, "(lane & 3) * 8 + (lane >> 2) * 2"),
          (4, "lane % 3 * 32 + lane // 3")]


def lane_words_expr(width, expr):
    return [eval(expr, {"__builtins__": {}}, {"lane": l}) * (width // 4) for l in range(32)]


def kernel_read_words(kind, warp, step, stage):
    import dense_fp32_tiled_gb300 as sg
    offs, width = sg.smem_request(kind, warp, step, stage)
    words = [o // 4 for o in offs]
    lo = min(words) // 64 * 64  # shift by a multiple of 64 words: every bank stays
    return width, [w - lo for w in words]


def patterns():
    """[(name, width, lane words)] in launch order."""
    out = [(f"{w} {e}", w, lane_words_expr(w, e)) for w, e in WIDE + NARROW]
    for kind, warp, step, stage, what in KERNEL_READS:
        w, words = kernel_read_words(kind, warp, step, stage)
        out.append((f"{w} kind{kind}:warp{warp}:step{step}:stage{stage}", w, words))
    return out


if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
    import dense_fp32_tiled_gb300 as sg
    from dense_fp32_tiled_gb300 import build
    build.build()
    sg.load_library()
    for i, (name, w, words) in enumerate(patterns()):
        assert all(0 <= x < 2048 and x % (w // 4) == 0 for x in words), name
        cyc, _ = sg.bank_pattern_probe(w, words)
        print(f"{i} {name} = {cyc:.3f} cycles per load")
