"""The bench's algorithmic work per op (the numerators of every roofline
fraction) against closed forms of the workloads, on the CPU.

Shapes, as the pages give them:
  - the LLaMA-2.4B-like IHA layer ("IHA-CUDA: Interleaved Head Attention
    Kernels for Hopper GPUs", "End-to-End Training Benchmark"): B=1, N=8192,
    H=20 heads, P=4 pseudo-heads per head, d=128, fp32 mixing weights [H,P,H];
  - its sliding-window attention ("FLOP Matching"): 80 pseudo-heads at
    N=4096 with W = WSL + 1 = 1024 keys per query including the diagonal;
  - the long-context layer: B=2, N=16384, causal over the 80 pseudo-heads;
  - Hiera-Base MAE stage 1 ("hiera-optim 0.1.0"): B=128, a 56x56 token grid
    of 8x8 mask units (49), 20 kept, C=96, one head.
Bytes count every input read once and every output written once (bf16
activations, fp32 weights, fp32 LSE, int32 keep ids); FLOPs count 2 per
multiply-add of the contractions the path defines.  The values are written
out here from those shapes, not taken from the bench's inputs, so a wrong
shape or a dropped term in the bench's table fails.

The last test keeps the ncu summaries under profiles/ reproducible: every
command they quote runs committed files, with flags the bench still takes,
and every ncu command leaves the GPU clocks alone.
"""
import glob
import os
import shlex
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

BF16, F32, I32 = 2, 4, 4


def _table():
    import bench
    return {name: (b, f) for name, b, f in bench.op_table()}


def _window_pairs(N: int, W: int) -> int:
    # query i sees keys max(0, i - W + 1) .. i: min(i + 1, W) of them
    return W * (W + 1) // 2 + (N - W) * W


def test_premix_layer_bytes_and_flops():
    B, N, H, P, d = 1, 8192, 20, 4, 128
    x = B * N * H * d * BF16            # 41.9 MB
    y = B * N * H * P * d * BF16        # 167.8 MB
    w = H * P * H * F32                 # 6.4 KB
    fl = 2 * B * N * (H * P) * H * d   # 3.36 GFLOP per tensor
    t = _table()
    assert (x, y, w) == (41_943_040, 167_772_160, 6_400)
    assert t["premix_fwd_qkv"] == (3 * (x + y + w), 3 * fl)
    # dX and dW of each tensor from one read of dY and X: dY + X in, dX + dW out
    assert t["premix_bwd_qkv"] == (3 * (y + 2 * x + 2 * w), 3 * 2 * fl)
    assert y + 2 * x + 2 * w == 251_671_040  # against 419.4 MB for two passes


def test_window_attention_flops_and_bytes():
    B, N, HP, d, W = 1, 4096, 80, 128, 1024
    pairs = _window_pairs(N, W)
    assert pairs == 3_670_528
    # brute force of the visible-pair count on a small case of the same rule
    n, win = 300, 37
    assert sum(1 for i in range(n) for j in range(n) if j <= i and i - j < win) == \
        _window_pairs(n, win)
    fl = 4 * d * pairs * HP * B        # QK^T and P.V: 2 * 2 * d per visible pair
    tens = B * N * HP * d * BF16
    lse = B * HP * N * F32
    t = _table()
    assert t["attention_window"] == (4 * tens + lse, fl)
    assert fl == 150_344_826_880
    # backward: Q, K, V, O, dO, lse in; dQ, dK, dV out; five contractions
    assert t["attention_window_bwd"] == (8 * tens + lse, fl * 5 // 2)


def test_long_context_layer():
    B, N, H, P, d = 2, 16384, 20, 4, 128
    x = B * N * H * d * BF16
    y = B * N * H * P * d * BF16
    w = H * P * H * F32
    t = _table()
    assert t["long_premix_fwd_qkv"] == (3 * (x + y + w), 3 * 2 * B * N * H * P * H * d)
    pairs = N * (N + 1) // 2           # causal
    fl = 4 * d * pairs * H * P * B
    assert fl == 10_995_787_366_400   # 11.0 TFLOP
    assert t["long_attention_causal"] == (4 * y + B * H * P * N * F32, fl)


def test_hiera_stage1_mask_units():
    B, keep, T, C = 128, 20, 64, 96
    kept = B * keep * T * C * BF16     # 31.5 MB of kept tokens
    ids = B * keep * I32
    t = _table()
    assert t["mu_gather"] == (2 * kept + ids, 0)
    assert t["mu_scatter"] == (2 * kept + ids, 0)
    assert t["mu_attention"] == (4 * kept, 4 * C * T * T * B * keep)
    assert 4 * C * T * T * B * keep == 4_026_531_840


def test_every_step_op_is_accounted():
    import bench
    names = [n for n, _, _ in bench.op_table()]
    assert sorted(names) == sorted([
        "premix_fwd_qkv", "premix_bwd_qkv", "attention_window", "attention_window_bwd",
        "mu_gather", "mu_attention", "mu_scatter", "long_premix_fwd_qkv",
        "long_attention_causal"])
    assert bench.launches_per_step() == 12


def _profile_commands():
    """Every command quoted in profiles/*.md (indented blocks, continuation
    lines joined), as (file, command) pairs."""
    out = []
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        lines = open(f).read().splitlines()
        block = []
        for ln in lines + [""]:
            if ln.startswith("    "):
                block.append(ln.strip())
            elif block:
                text = " ".join(b[:-1].strip() if b.endswith("\\") else b for b in block)
                out += [(f, c.strip()) for c in text.split("&&") if c.strip()]
                block = []
    return out


def _committed(path: str) -> bool:
    r = subprocess.run(["git", "ls-files", "--error-unmatch", path], cwd=ROOT,
                       capture_output=True, text=True)
    if r.returncode == 0:
        return True
    inside = subprocess.run(["git", "rev-parse", "--is-inside-work-tree"], cwd=ROOT,
                            capture_output=True, text=True)
    # outside a git checkout (an exported tree): the file must at least exist
    return inside.returncode != 0 and os.path.exists(os.path.join(ROOT, path))


def test_profile_commands_run_committed_files_with_current_flags():
    import bench
    cmds = _profile_commands()
    files = {os.path.basename(f) for f, _ in cmds}
    assert files == {os.path.basename(f) for f in glob.glob(os.path.join(ROOT, "profiles", "*.md"))}
    ap = bench.make_parser()
    for f, c in cmds:
        argv = shlex.split(c)
        assert "_work" not in c, (f, c)
        if argv[0] == "ncu":
            assert "--clock-control" in argv and argv[argv.index("--clock-control") + 1] == "none", (f, c)
        if "bench.py" in argv:
            rest = argv[argv.index("bench.py") + 1:]
            try:
                ap.parse_args(rest)
            except SystemExit:
                raise AssertionError(f"{os.path.basename(f)}: bench.py {' '.join(rest)}")
        for a in argv:
            if a.endswith(".py") and not a.startswith("-"):
                assert _committed(a), (f, a)
