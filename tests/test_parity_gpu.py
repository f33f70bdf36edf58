"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Cases follow the operator's own test grid (ONNX Runtime PR #33384, "Testing"):
the real shape 4 x 2560, rank 320, for fp32 / fp16 / bf16, several row
counts, with and without the prologue; small and irregular shapes; default and
non-default attributes; two chained blocks; bitwise row independence;
streams_out pass-through; zero rows; CUDA-graph capture and replay bitwise
equal to eager. Plus determinism over repeated runs, guard bands around every
output, and misaligned pointers.
"""
import numpy as np
import pytest
import torch

from _parity import KEYS, compare, run_gpu, run_oracle
from _util import TORCH_DT, to_codes
from hyper_connection_rank_gb300 import inputs as I

pytestmark = pytest.mark.gpu

DEFAULT_ATTRS = dict(epsilon=1e-5, reduction_scale=1.0, silu_alpha=1.0, gate_div=1.0, gate_mul=1.0)
ODD_ATTRS = dict(epsilon=0.5, reduction_scale=1.5, silu_alpha=2.0, gate_div=0.7, gate_mul=3.0)


@pytest.fixture(scope="module")
def hc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import hyper_connection_rank_gb300 as m
    m.debug_wait_timeouts(reset=True)
    yield m
    assert m.debug_wait_timeouts() == 0, "a bounded device wait gave up"


def check(hc, rows, C, H, R, dt, prologue=True, attrs=I.QWEN_ATTRS, seed=0, flags=0, expect_path=None):
    d = I.make_block(rows, C, H, R, dt, seed=seed, prologue=prologue)
    if expect_path is not None:
        assert hc.path(rows, C, H, R, TORCH_DT[dt], flags) == expect_path
    gpu = run_gpu(hc, d, C, attrs, flags=flags)
    ref = run_oracle(d, C, dt, attrs)
    return compare(gpu, ref, dt, C, H, R, attrs, inputs=d)


# ------------------------------------------------------------ tiny config --

@pytest.mark.parametrize("flags", [0, 2], ids=["auto", "general"])
def test_tiny_fp32_block(hc, flags):
    """rows=2, C=4, H=64, R=16, fp32, no prologue, Qwen attributes, seed 0."""
    check(hc, 2, 4, 64, 16, "f32", prologue=False, flags=flags)


# --------------------------------------------------- real shape, decode rows --

@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("prologue", [True, False])
def test_real_shape_decode(hc, dt, rows, prologue):
    st = check(hc, rows, 4, 2560, 320, dt, prologue=prologue, expect_path=hc.HC_PATH_DECODE)
    print(dt, rows, prologue, st)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("rows", [1, 8])
def test_second_prefill_shape_decode_rows(hc, dt, rows):
    """C=8, H=1280, R=320 (the second prefill shape) at decode row counts."""
    check(hc, rows, 8, 1280, 320, dt, expect_path=hc.HC_PATH_DECODE)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("rows", [2, 5])
@pytest.mark.parametrize("shape", [(8, 1280, 200), (4, 1024, 104)], ids=lambda s: "C%d_H%d_R%d" % s)
def test_decode_ranks_with_ragged_column_shares(hc, dt, rows, shape):
    """Decode with two or more rows hands each up rank a share of ceil(R/C)
    (rounded to 4) down columns; with these R the last rank's share is short
    (4 and 20 columns): every column still reaches its consumer."""
    C, H, R = shape
    check(hc, rows, C, H, R, dt, seed=21, expect_path=hc.HC_PATH_DECODE)


@pytest.mark.parametrize("attrs", [DEFAULT_ATTRS, ODD_ATTRS], ids=["default", "odd"])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_attributes(hc, attrs, dt):
    check(hc, 3, 4, 2560, 320, dt, attrs=attrs)


# ------------------------------------------------- small / irregular shapes --

SHAPES = [(1, 64, 8), (2, 32, 16), (3, 40, 24), (4, 64, 16), (8, 32, 32), (4, 4096, 512), (1, 4096, 64),
          (2, 1000, 33), (8, 128, 512), (2, 96, 40), (4, 640, 168)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "C%d_H%d_R%d" % s)
@pytest.mark.parametrize("rows", [1, 7])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_small_and_irregular_shapes(hc, shape, rows, dt):
    C, H, R = shape
    check(hc, rows, C, H, R, dt, seed=3)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("rows", [9, 12, 16])
def test_real_shape_decode_up_to_16_rows(hc, dt, rows):
    """The tensor-core decode pair serves up to 16 rows (the MMA's N) where a
    CTA of each kernel still shares an SM at 16 rows: C = 4, H = 2560 does
    (decode at 9-16 rows), C = 8, H = 1280 does not (prefill from 9 rows)."""
    check(hc, rows, 4, 2560, 320, dt, expect_path=hc.HC_PATH_DECODE)
    check(hc, rows, 8, 1280, 320, dt, seed=3, expect_path=hc.HC_PATH_PREFILL)


# ---------------------------------------------- general path, more rows --

@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows", [9, 16, 128])
def test_real_shape_more_rows(hc, dt, rows):
    check(hc, rows, 4, 2560, 320, dt)


@pytest.mark.parametrize("dt,C,H", [("bf16", 4, 2560), ("f16", 8, 1280)])
def test_prefill_full_size_every_row(hc, dt, C, H):
    """rows = 8192 at the two prefill shapes, every row against the oracle
    (which runs its rows in parallel on the host cores), in chunks of 1024
    rows so the oracle's per-row trace stays small."""
    rows, R, chunk = 8192, 320, 1024
    d = I.make_block(rows, C, H, R, dt, seed=0, prologue=True)
    gpre, gpost, gsout = run_gpu(hc, d, C, I.QWEN_ATTRS)
    for lo in range(0, rows, chunk):
        hi = min(rows, lo + chunk)
        ref = run_oracle(d, C, dt, I.QWEN_ATTRS, rows_idx=torch.arange(lo, hi))
        compare((gpre[lo:hi], gpost[lo:hi], gsout[lo:hi]), ref, dt, C, H, R, I.QWEN_ATTRS, inputs=d)


# ----------------------------------------------------------- invariants --

@pytest.mark.parametrize("rows,flags", [(8, 0), (16, 0), (8, 2), (40, 2)],
                         ids=["decode", "decode16", "general", "general40"])
def test_row_independence_bitwise(hc, rows, flags):
    """A row gives the same bits at any batch size, within one path."""
    C, H, R = 4, 2560, 320
    d = I.make_block(rows, C, H, R, "bf16", seed=5, prologue=True)
    full = run_gpu(hc, d, C, I.QWEN_ATTRS, flags=flags)
    for j in (0, rows // 2, rows - 1):
        one = {k: (v[j:j + 1] if k in ("streams", "prev_out", "prev_gate") else v) for k, v in d.items()}
        r = run_gpu(hc, one, C, I.QWEN_ATTRS, flags=flags)
        for a, b in zip(full, r):
            assert np.array_equal(a[j:j + 1], b)


@pytest.mark.parametrize("rows,flags", [(1, 0), (8, 0), (16, 0), (4, 2), (300, 0)])
def test_deterministic_over_20_runs(hc, rows, flags):
    d = I.make_block(rows, 4, 2560, 320, "bf16", seed=6, prologue=True)
    first = run_gpu(hc, d, 4, I.QWEN_ATTRS, flags=flags)
    for _ in range(19):
        again = run_gpu(hc, d, 4, I.QWEN_ATTRS, flags=flags)
        for a, b in zip(first, again):
            assert np.array_equal(a, b)


def test_streams_out_passthrough_and_optional(hc):
    d = I.make_block(3, 4, 2560, 320, "bf16", seed=7, prologue=False)
    pre, post, sout = run_gpu(hc, d, 4, I.QWEN_ATTRS)
    assert np.array_equal(sout, to_codes(d["streams"]))
    pre2, post2, none = run_gpu(hc, d, 4, I.QWEN_ATTRS, want_streams_out=False)
    assert none is None and np.array_equal(pre, pre2) and np.array_equal(post, post2)


def test_prefill_mid_reduction_variants_same_bits(hc):
    """Batches of up to 64 rows sum the K-slice partials with one thread per
    column, larger ones with one per four columns: the same additions in the
    same order, so the rows of a 40-row call equal the same rows of a 100-row
    call bit for bit."""
    C, H, R = 4, 2560, 320
    d = I.make_block(100, C, H, R, "bf16", seed=41, prologue=True)
    full = run_gpu(hc, d, C, I.QWEN_ATTRS)
    sub = {k: (v[30:70] if k in ("streams", "prev_out", "prev_gate") else v) for k, v in d.items()}
    part = run_gpu(hc, sub, C, I.QWEN_ATTRS)
    for a, b in zip(full, part):
        assert np.array_equal(a[30:70], b)


@pytest.mark.parametrize("rows", [300, 700])
def test_prefill_without_streams_out_bitwise(hc, rows):
    """With no streams_out requested the prefill path gives pre_output and
    post_gate the same bits as with it, in both K-split regimes (300 rows:
    256-wide slices; 700 rows: branch-sized slices)."""
    d = I.make_block(rows, 4, 2560, 320, "bf16", seed=37, prologue=True)
    assert hc.path(rows, 4, 2560, 320, torch.bfloat16) == hc.HC_PATH_PREFILL
    pre, post, sout = run_gpu(hc, d, 4, I.QWEN_ATTRS)
    pre2, post2, none = run_gpu(hc, d, 4, I.QWEN_ATTRS, want_streams_out=False)
    assert none is None and np.array_equal(pre, pre2) and np.array_equal(post, post2)


def test_zero_up_and_inject_weights(hc):
    d = I.make_block(2, 4, 2560, 320, "bf16", seed=8, prologue=True)
    d["up_w"] = torch.zeros_like(d["up_w"])
    d["inject_w"] = torch.zeros_like(d["inject_w"])
    gpu = run_gpu(hc, d, 4, I.QWEN_ATTRS)
    compare(gpu, run_oracle(d, 4, "bf16", I.QWEN_ATTRS), "bf16", 4, 2560, 320, I.QWEN_ATTRS, inputs=d)
    post = torch.from_numpy(gpu[1].view(np.int16)).view(torch.bfloat16).float()
    assert torch.all(post == 1.0)  # gate_mul / 2


def test_zero_rows(hc):
    d = I.make_block(0, 4, 2560, 320, "bf16", seed=0, prologue=True)
    pre, post, sout = run_gpu(hc, d, 4, I.QWEN_ATTRS)
    assert pre.shape == (0, 2560) and post.shape == (0, 4) and sout.shape == (0, 10240)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_two_chained_blocks(hc, dt):
    """Block 2's prologue takes block 1's pre_output and post_gate, and its
    streams are block 1's streams_out; each side runs its own chain."""
    C, H, R, rows = 4, 2560, 320, 2
    d1 = I.make_block(rows, C, H, R, dt, seed=9, block=0, prologue=True)
    w2 = I.make_weights(C, H, R, dt, seed=9, block=1)
    g1 = run_gpu(hc, d1, C, I.QWEN_ATTRS)
    o1 = run_oracle(d1, C, dt, I.QWEN_ATTRS)
    compare(g1, o1, dt, C, H, R, I.QWEN_ATTRS, inputs=d1)
    from _util import from_codes
    g2 = run_gpu(hc, dict(w2, streams=from_codes(g1[2], dt), prev_out=from_codes(g1[0], dt),
                          prev_gate=from_codes(g1[1], dt)), C, I.QWEN_ATTRS)
    o2 = run_oracle(dict(w2, streams=from_codes(o1[2], dt), prev_out=from_codes(o1[0], dt),
                         prev_gate=from_codes(o1[1], dt)), C, dt, I.QWEN_ATTRS)
    compare(g2, o2, dt, C, H, R, I.QWEN_ATTRS, check_streams_out=False, inputs=w2)


def test_decode_chain_under_pdl_matches_oracle_block_by_block(hc):
    """The 96-block decode chain as the benchmark launches it: rows 1, bf16,
    96 distinct weight sets, every block enqueued back to back on one stream
    with the weights-static flag and one shared workspace, so each block's
    kernels start while the previous block's still run (programmatic
    dependent launch). Every block keeps its outputs; block i is checked
    against the oracle fed with the GPU's own inputs to block i (block i-1's
    outputs), so a read of data the previous block had not yet written, or a
    workspace reused too early, shows as a mismatch."""
    C, H, R, rows, n = 4, 2560, 320, 1, 96
    dev = torch.device("cuda")
    flags = hc.HC_FLAG_WEIGHTS_STATIC
    weights = [I.make_weights(C, H, R, "bf16", seed=0, block=i, device=dev) for i in range(n)]
    a0 = I.make_activations(rows, C, H, "bf16", seed=0, block=0, prologue=True, device=dev)
    pre = torch.empty(n, rows, H, dtype=torch.bfloat16, device=dev)
    post = torch.empty(n, rows, C, dtype=torch.bfloat16, device=dev)
    sout = torch.empty(n, rows, C * H, dtype=torch.bfloat16, device=dev)
    work = torch.empty(max(1, hc.workspace_size(rows, C, H, R, torch.bfloat16, flags)), dtype=torch.uint8, device=dev)

    def inputs_of(i):
        if i == 0:
            return a0["streams"], a0["prev_out"], a0["prev_gate"]
        return sout[i - 1], pre[i - 1], post[i - 1]

    for i in range(n):
        st, po, pg = inputs_of(i)
        w = weights[i]
        hc.lowrank_mix(st, w["norm_scale"], w["down_w"], w["up_w"], w["inject_w"], po, pg, num_branches=C,
                       flags=flags, out=(pre[i], post[i], sout[i]), workspace=work, **I.QWEN_ATTRS)
    torch.cuda.synchronize()
    assert torch.isfinite(pre.float()).all() and torch.isfinite(post.float()).all()
    for i in range(n):
        st, po, pg = inputs_of(i)
        d = {k: v.cpu() for k, v in weights[i].items()}
        d.update(streams=st.cpu(), prev_out=po.cpu(), prev_gate=pg.cpu())
        ref = run_oracle(d, C, "bf16", I.QWEN_ATTRS)
        gpu = (to_codes(pre[i]), to_codes(post[i]), to_codes(sout[i]))
        compare(gpu, ref, "bf16", C, H, R, I.QWEN_ATTRS, inputs=d)


@pytest.mark.parametrize("rows", [1, 8, 64])
def test_cuda_graph_replay_bitwise_equal_to_eager(hc, rows):
    C, H, R = 4, 2560, 320
    d = I.make_block(rows, C, H, R, "bf16", seed=10, prologue=True)
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    eager = hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, **I.QWEN_ATTRS)
    torch.cuda.synchronize()
    pre = torch.empty_like(eager[0]); post = torch.empty_like(eager[1]); sout = torch.empty_like(eager[2])
    ws = torch.empty(hc.workspace_size(rows, C, H, R, torch.bfloat16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, out=(pre, post, sout), workspace=ws,
                           **I.QWEN_ATTRS)
    for _ in range(3):
        pre.zero_(); post.zero_(); sout.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, (pre, post, sout)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_guard_bands_untouched(hc):
    """Outputs and workspace sit inside larger buffers filled with a sentinel;
    the bytes around them must survive the call (stands in for memcheck)."""
    C, H, R = 4, 2560, 320
    for rows, flags in ((3, 0), (3, 2), (20, 0)):
        d = I.make_block(rows, C, H, R, "bf16", seed=11, prologue=True)
        g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
        pad = 4096

        def guarded(n):
            buf = torch.full((n + 2 * pad,), 0x5A5A, dtype=torch.int16, device="cuda")
            return buf, buf[pad:pad + n].view(torch.bfloat16)

        bp, pre = guarded(rows * H)
        bq, post = guarded(rows * C)
        bs, sout = guarded(rows * C * H)
        nws = hc.workspace_size(rows, C, H, R, torch.bfloat16, flags)
        wbuf = torch.full((nws + 2 * 8192,), 0xA5, dtype=torch.uint8, device="cuda")
        ws = wbuf[8192:8192 + nws]
        hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, out=(pre.view(rows, H), post.view(rows, C),
                                                                    sout.view(rows, C * H)),
                       workspace=ws, flags=flags, **I.QWEN_ATTRS)
        torch.cuda.synchronize()
        for buf, n in ((bp, rows * H), (bq, rows * C), (bs, rows * C * H)):
            assert torch.all(buf[:pad] == 0x5A5A) and torch.all(buf[pad + n:] == 0x5A5A)
        assert torch.all(wbuf[:8192] == 0xA5) and torch.all(wbuf[8192 + nws:] == 0xA5)


@pytest.mark.parametrize("rows,dt,flags", [(1, "bf16", 0), (5, "bf16", 0), (5, "f32", 0), (300, "bf16", 0),
                                            (600, "f16", 0), (5, "bf16", 2), (40, "f32", 2)],
                         ids=["decode1", "decode5", "decode5-f32", "prefill300", "prefill600-f16", "general5",
                              "general40-f32"])
def test_workspace_poisoned_with_nan(hc, rows, dt, flags):
    """Every path writes each workspace word before reading it: a workspace
    filled with NaN bytes and one filled with zeros give bitwise the same
    outputs (a read of stale scratch would carry the NaN into them)."""
    C, H, R = 4, 2560, 320
    d = I.make_block(rows, C, H, R, dt, seed=43, prologue=True)
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    n = hc.workspace_size(rows, C, H, R, TORCH_DT[dt], flags)
    outs = []
    for fill in (0xFF, 0x00):
        ws = torch.full((max(n, 1),), fill, dtype=torch.uint8, device="cuda")
        outs.append(hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, workspace=ws, flags=flags,
                                   **I.QWEN_ATTRS))
        torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert not torch.isnan(outs[0][0].float()).any() and not torch.isnan(outs[0][1].float()).any()


def test_misaligned_pointers_take_general_path(hc):
    C, H, R, rows = 4, 256, 32, 3
    d = I.make_block(rows, C, H, R, "bf16", seed=12, prologue=True)
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    big = torch.empty(rows * C * H + 1, dtype=torch.bfloat16, device="cuda")
    st = big[1:].view(rows, C * H)          # 2-byte offset: not 16-byte aligned
    st.copy_(g["streams"])
    out = hc.lowrank_mix(st, *[g[k] for k in KEYS[1:]], num_branches=C, **I.QWEN_ATTRS)
    torch.cuda.synchronize()
    ref = run_oracle(d, C, "bf16", I.QWEN_ATTRS)
    compare(tuple(to_codes(t) for t in out), ref, "bf16", C, H, R, I.QWEN_ATTRS, inputs=d)


def test_workspace_errors(hc):
    C, H, R, rows = 4, 2560, 320, 2
    d = I.make_block(rows, C, H, R, "bf16", seed=0, prologue=True)
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    need = hc.workspace_size(rows, C, H, R, torch.bfloat16)
    assert need > 256
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(hc.HcError) as e:
        hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, workspace=small, **I.QWEN_ATTRS)
    assert e.value.status == 3


@pytest.mark.parametrize("small,large,dt", [(16, 17, "bf16"), (16, 17, "f16"), (512, 513, "bf16"), (512, 513, "f16")],
                         ids=["decode8-prefill9-bf16", "decode8-prefill9-f16", "prefill512-513-bf16",
                              "prefill512-513-f16"])
def test_row_bits_across_batch_size_switches(hc, small, large, dt):
    """The same rows in a batch just below and just above a switch of the
    path (16 -> 17 rows: decode -> prefill) or of the prefill path's K split
    (512 -> 513 rows: 256-wide slices -> branch-wide slices). Both sides meet
    the oracle tolerance (tested above); here the difference between them is
    measured and bounded: streams_out identical, most pre_output elements
    bit-identical, the histogram of ulp distances appended to HC_PARITY_LOG."""
    import json
    import os
    from _util import ulp_diff
    C, H, R = 4, 2560, 320
    d = I.make_block(large, C, H, R, dt, seed=47, prologue=True)
    sub = {k: (v[:small] if k in ("streams", "prev_out", "prev_gate") else v) for k, v in d.items()}
    a = run_gpu(hc, sub, C, I.QWEN_ATTRS)
    b = run_gpu(hc, d, C, I.QWEN_ATTRS)
    assert np.array_equal(a[2], b[2][:small])
    up = ulp_diff(a[0], b[0][:small], dt)
    uq = ulp_diff(a[1], b[1][:small], dt)
    hist = {str(k): int((up == k).sum()) for k in range(4)}
    hist[">3"] = int((up > 3).sum())
    rec = {"kind": "batch_size_switch", "rows": [small, large], "dtype": dt,
           "paths": [hc.PATH_NAMES[hc.path(n, C, H, R, TORCH_DT[dt])] for n in (small, large)],
           "pre_identical": float((up == 0).mean()), "pre_ulp_hist": hist, "pre_max_ulp": int(up.max()),
           "post_identical": float((uq == 0).mean()), "post_max_ulp": int(uq.max())}
    path = os.environ.get("HC_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    print(rec)
    assert rec["pre_identical"] >= 0.8 and rec["post_max_ulp"] <= 2


def test_cross_path_agreement(hc):
    """Decode and general paths accumulate in different orders; both meet the
    oracle tolerance, and they agree with each other on most elements."""
    d = I.make_block(4, 4, 2560, 320, "bf16", seed=13, prologue=True)
    a = run_gpu(hc, d, 4, I.QWEN_ATTRS, flags=0)
    b = run_gpu(hc, d, 4, I.QWEN_ATTRS, flags=2)
    assert np.array_equal(a[2], b[2])
    assert (a[0] == b[0]).mean() > 0.8


@pytest.mark.parametrize("rows,dt,flags", [(5, "bf16", 0), (5, "f16", 0), (5, "f32", 0), (130, "bf16", 0),
                                            (130, "f16", 0), (5, "bf16", 2), (5, "f32", 2)],
                         ids=["decode-bf16", "decode-f16", "decode-f32", "prefill-bf16", "prefill-f16",
                              "general-bf16", "general-f32"])
def test_special_values(hc, rows, dt, flags):
    """IEEE special values on every path, against the oracle: a NaN in one
    branch of row 1's streams and an inf in row 2's prev_out make those rows'
    pre_output and post_gate NaN (streams_out keeps them only where they
    entered); in row 3 (fp32 / bf16) one branch overflows its sum of squares,
    so its inv is 0 and its hn zero, a finite result held to the usual
    tolerance; the other rows are unaffected."""
    C, H, R = 4, 2560, 320
    d = I.make_block(rows, C, H, R, dt, seed=41, prologue=True)
    d["streams"][1, 1 * H + 5] = float("nan")
    d["prev_out"][2, 7] = float("inf")
    if dt != "f16":
        v = d["streams"].view(rows, C, H)
        v[3, 2] = (v[3, 2].double() * 2.0 ** 100).to(TORCH_DT[dt])
    path = {0: None, 2: hc.HC_PATH_GENERAL}[flags]
    if path is not None:
        assert hc.path(rows, C, H, R, TORCH_DT[dt], flags) == path
    gpre, gpost, gsout = run_gpu(hc, d, C, I.QWEN_ATTRS, flags=flags)
    opre, opost, osout, _ = run_oracle(d, C, dt, I.QWEN_ATTRS)
    from _util import codes_to_f64
    for g, o in ((gpre, opre), (gpost, opost)):
        gn, on = np.isnan(codes_to_f64(g, dt)), np.isnan(codes_to_f64(o, dt))
        assert np.array_equal(gn, on)
        assert on[1:3].all() and not on[[0] + list(range(3, rows))].any()
    gs, os_ = codes_to_f64(gsout, dt), codes_to_f64(osout, dt)
    assert np.array_equal(np.isnan(gs), np.isnan(os_)) and np.isnan(os_).sum() == 1
    fin = ~np.isnan(os_)
    assert np.array_equal(gs[fin], os_[fin]) and np.isinf(os_).sum() == C
    keep = torch.tensor([0] + list(range(3, rows)))
    ref = run_oracle(d, C, dt, I.QWEN_ATTRS, rows_idx=keep)
    k = keep.numpy()
    compare((gpre[k], gpost[k], gsout[k]), ref, dt, C, H, R, I.QWEN_ATTRS, inputs=d)


# ------------------------------------------------- prefill (tensor cores) --

PREFILL_SHAPES = [(4, 2560, 320), (8, 1280, 320), (1, 4096, 64), (2, 128, 64), (8, 64, 128), (4, 256, 448),
                  (1, 16384, 64)]  # the last: a 64 KB row for the norm kernel


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=lambda s: "C%d_H%d_R%d" % s)
@pytest.mark.parametrize("rows", [17, 130, 300])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_prefill_path_shapes(hc, shape, rows, dt):
    """tcgen05 path: one partial tile, several tiles with a ragged tail."""
    C, H, R = shape
    check(hc, rows, C, H, R, dt, seed=17, expect_path=hc.HC_PATH_PREFILL)


@pytest.mark.parametrize("prologue", [True, False])
@pytest.mark.parametrize("attrs", [I.QWEN_ATTRS, ODD_ATTRS], ids=["qwen", "odd"])
def test_prefill_attributes_and_prologue(hc, prologue, attrs):
    check(hc, 200, 4, 2560, 320, "bf16", prologue=prologue, attrs=attrs, expect_path=hc.HC_PATH_PREFILL)


def test_prefill_large_batch_regime(hc):
    """Past 512 rows the prefill path splits K by branch (below, 256 wide):
    parity at 600 rows, and a row's bits equal in calls of 640 and 530 rows
    (both in that regime)."""
    C, H, R = 4, 2560, 320
    check(hc, 600, C, H, R, "bf16", seed=23, expect_path=hc.HC_PATH_PREFILL)
    d = I.make_block(640, C, H, R, "bf16", seed=29, prologue=True)
    full = run_gpu(hc, d, C, I.QWEN_ATTRS)
    for lo, hi in ((0, 530), (110, 640)):
        sub = {k: (v[lo:hi] if k in ("streams", "prev_out", "prev_gate") else v) for k, v in d.items()}
        part = run_gpu(hc, sub, C, I.QWEN_ATTRS)
        for a, b in zip(full, part):
            assert np.array_equal(a[lo:hi], b)


@pytest.mark.parametrize("dt,C,H", [("bf16", 4, 2560), ("f16", 4, 2560), ("bf16", 8, 1280), ("f16", 8, 1280)])
def test_prefill_full_size_deterministic(hc, dt, C, H):
    """Repeated 8192-row calls give identical bits in both 16-bit types (a
    race between a consumer's reads and a producer's refill shows here first)."""
    d = I.make_block(8192, C, H, 320, dt, seed=37, prologue=True)
    first = run_gpu(hc, d, C, I.QWEN_ATTRS)
    for _ in range(4):
        again = run_gpu(hc, d, C, I.QWEN_ATTRS)
        for a, b in zip(first, again):
            assert np.array_equal(a, b)


@pytest.mark.parametrize("dt,C,H", [("bf16", 4, 2560), ("f16", 8, 1280)])
def test_prefill_full_size_row_invariance(hc, dt, C, H):
    """At the 8192-row prefill shapes every output of a row is bitwise the
    same in the full call and in calls on two sub-batches (other tile
    positions, other CTAs, a ragged last tile): catches any exchange between
    rows, including a producer that overwrites a buffer a consumer still reads."""
    R = 320
    d = I.make_block(8192, C, H, R, dt, seed=31, prologue=True)
    full = run_gpu(hc, d, C, I.QWEN_ATTRS)
    for lo, hi in ((0, 4096), (1000, 8192)):
        sub = {k: (v[lo:hi] if k in ("streams", "prev_out", "prev_gate") else v) for k, v in d.items()}
        part = run_gpu(hc, sub, C, I.QWEN_ATTRS)
        for a, b in zip(full, part):
            assert np.array_equal(a[lo:hi], b)


def test_prefill_row_independence_bitwise(hc):
    """Within the prefill path a row's bits do not depend on the batch: rows
    of a 300-row call equal the same rows in 137- and 150-row calls (different
    tile positions)."""
    C, H, R = 4, 2560, 320
    d = I.make_block(300, C, H, R, "bf16", seed=19, prologue=True)
    full = run_gpu(hc, d, C, I.QWEN_ATTRS)
    for lo, hi in ((0, 137), (150, 300), (7, 160)):
        sub = {k: (v[lo:hi] if k in ("streams", "prev_out", "prev_gate") else v) for k, v in d.items()}
        part = run_gpu(hc, sub, C, I.QWEN_ATTRS)
        for a, b in zip(full, part):
            assert np.array_equal(a[lo:hi], b)
