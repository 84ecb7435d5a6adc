"""GPU checks of gdn_prefill_chunked, the tensor-core chunked form of the
rule over many tokens a sequence ("mstar PR #965", "Correctness": the
chunked GDN path; "mstar PR #1127": one GDN prefill kernel).

1. Against the fp64 oracle (the rule token after token): every output within
   the bf16 tolerance, every final state within the chained-state tolerance;
   sequences of 1, 63, 64, 65, 130 and 512 tokens cover whole chunks, ragged
   tails and one-token chunks, and last chunks of 17, 31, 48 and 49 tokens
   end inside or at the edge of a 16-token row block; in place and twin,
   the 0.8B and 9B (grouped heads) shapes, bf16 and fp32 activations.
2. Against the exact token-serial gdn_prefill on the GPU: the two agree far
   inside the tolerances (about 1e-5 relative), so the chunking adds no
   error the oracle tolerances would hide.
3. Padding, empty, bad slots and bad token ranges behave as in gdn_prefill,
   bit for bit: zero outputs, untouched slots, the device error word.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_decode_gb300 import inputs as I
from gpu_helpers import STATE_TOL_CHAIN, assert_out_close, f64, state_rel_err, ti
from test_gpu_prefill import Case

pytestmark = pytest.mark.gpu


def chunked(c, keep_in_place=False, out=None):
    return c.gdn.gdn_prefill_chunked(c.dev["q"], c.dev["k"], c.dev["v"], c.dev["a"], c.dev["b"], c.A_log,
                                     c.dt_bias, c.pool, c.cu, c.rs, None if keep_in_place else c.ws,
                                     out=out, keep_in_place=keep_in_place)


def oracle(orc, c, keep_in_place):
    pool = c.pool_np.astype(np.float64).copy()
    o_ref, bad = orc.prefill(c.cu_np, c.ref["q"], c.ref["k"], c.ref["v"], c.ref["a"], c.ref["b"],
                             c.prm["A_log"], c.prm["dt_bias"], pool, c.rs_np,
                             write_slot=None if keep_in_place else c.ws_np)
    assert bad == 0
    return o_ref, pool


def check_against_oracle(c, out, o_ref, pool, keep_in_place):
    assert_out_close(f64(out), o_ref, c.s.dtype)
    got = c.pool.tensor.cpu().numpy()
    real = c.rs_np > 0
    slots = c.rs_np[real] if keep_in_place else c.ws_np[real]
    for sl in slots:
        for h in range(c.s.hv):
            err = state_rel_err(got[sl, h], pool[sl, h])
            assert err <= STATE_TOL_CHAIN, f"slot {sl} head {h}: {err:.3g}"
    # every slot no real sequence writes is untouched (padding's included)
    written = set(int(x) for x in slots)
    for sl in range(c.num_slots):
        if sl not in written:
            assert np.array_equal(got[sl], c.pool_np[sl]), f"slot {sl} changed"


CASES = [(I.QWEN_08B, [130, 64, 0, 1, 63, 65]), (I.QWEN_9B, [70, 0, 129, 5]),
         (I.QWEN_08B.with_(dtype="f32"), [65, 3, 128]),
         # last chunks ending inside or at the edge of a chunk's 16-token row
         # blocks (17, 48, 31 and 49 tokens)
         (I.QWEN_08B, [17, 112, 95, 49])]
IDS = ["0.8b", "9b", "0.8b-f32", "0.8b-row-block-tails"]


@pytest.mark.parametrize("shape,lens", CASES, ids=IDS)
@pytest.mark.parametrize("keep_in_place", [False, True], ids=["twin", "in_place"])
def test_chunked_matches_oracle(gdn, orc, shape, lens, keep_in_place):
    c = Case(gdn, shape, lens, seed=90)
    out = chunked(c, keep_in_place)
    torch.cuda.synchronize()
    o_ref, pool = oracle(orc, c, keep_in_place)
    check_against_oracle(c, out, o_ref, pool, keep_in_place)
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_chunked_512_tokens_matches_oracle(gdn, orc):
    """Eight chunks in one sequence (0.8B shape, twin) against the oracle."""
    c = Case(gdn, I.QWEN_08B, [512, 0, 200], seed=91, n_pad=0)
    out = chunked(c)
    torch.cuda.synchronize()
    o_ref, pool = oracle(orc, c, False)
    check_against_oracle(c, out, o_ref, pool, False)
    assert gdn.get_device_error() == 0


@pytest.mark.parametrize("shape,lens", [(I.QWEN_08B, [512, 97, 0, 64, 1]), (I.QWEN_9B, [300, 33])],
                         ids=["0.8b", "9b"])
def test_chunked_close_to_exact_prefill(gdn, shape, lens):
    """The chunked and the token-serial kernels on the same inputs: states
    within 5e-5 of each other (relative to each head's largest entry), fp32
    outputs of the same kernels likewise."""
    for dtype in ("bf16", "f32"):
        s = shape.with_(dtype=dtype)
        c = Case(gdn, s, lens, seed=92)
        ref = c.prefill().clone()
        torch.cuda.synchronize()
        ref_pool = c.pool.tensor.clone()
        c.reset()
        out = chunked(c)
        torch.cuda.synchronize()
        got, want = c.pool.tensor.cpu().numpy(), ref_pool.cpu().numpy()
        for sl in c.ws_np[c.rs_np > 0]:
            for h in range(s.hv):
                err = state_rel_err(got[sl, h], want[sl, h].astype(np.float64))
                assert err <= 5e-5, f"{dtype} slot {sl} head {h}: {err:.3g}"
        if dtype == "f32":
            o, r = f64(out), f64(ref)
            scale = np.abs(r).max()
            assert np.abs(o - r).max() <= 5e-5 * scale
        else:
            assert_out_close(f64(out), f64(ref), "bf16")
    assert gdn.get_device_error() == 0


def test_chunked_padding_bad_slots_and_ranges(gdn):
    """The same sequence-level contract as gdn_prefill, bit for bit."""
    s = I.QWEN_08B
    # a bad write slot (equal to the read slot) spoils that sequence only
    c = Case(gdn, s, [70, 3, 5], seed=93, n_pad=0)
    start = torch.from_numpy(c.pool_np).cuda()
    ws = c.ws_np.copy()
    ws[1] = c.rs_np[1]
    c.ws = ti(ws)
    out = chunked(c)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 1
    assert not out[c.cu_np[1]:c.cu_np[2]].any()
    assert out[c.cu_np[0]:c.cu_np[1]].any()
    assert torch.equal(c.pool.tensor[int(c.rs_np[1])], start[int(c.rs_np[1])])
    # a token range past total_tokens is bad; the other sequences run
    c.reset()
    c.ws = ti(c.ws_np)
    cu = c.cu_np.copy()
    cu[3] = c.T + 5
    c.cu = ti(cu)
    out = chunked(c)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 1
    assert torch.equal(c.pool.tensor[int(c.ws_np[2])], start[int(c.ws_np[2])])
    assert not torch.equal(c.pool.tensor[int(c.ws_np[0])], start[int(c.ws_np[0])])
    # padding rows (read slot 0) write zeros and touch nothing; an empty twin
    # sequence moves its state unchanged
    c2 = Case(gdn, s, [0, 2, 66], seed=94, n_pad=1)
    start2 = torch.from_numpy(c2.pool_np).cuda()
    out = torch.full((c2.T, s.hv, s.dv), 7.0, dtype=torch.bfloat16, device="cuda")
    chunked(c2, out=out)
    torch.cuda.synchronize()
    assert torch.equal(c2.pool.tensor[int(c2.ws_np[0])], start2[int(c2.rs_np[0])])
    for r in range(len(c2.lens)):
        if c2.rs_np[r] == 0:
            assert not out[c2.cu_np[r]:c2.cu_np[r + 1]].any()
    assert gdn.get_device_error() == 0


def test_chunked_in_place_equals_twin(gdn):
    """In place and twin run the same arithmetic: identical outputs and states."""
    c = Case(gdn, I.QWEN_08B, [150, 7, 64], seed=95, n_pad=0)
    out_t = chunked(c).clone()
    torch.cuda.synchronize()
    twin = c.pool.tensor.clone()
    c.reset()
    out_i = chunked(c, keep_in_place=True)
    torch.cuda.synchronize()
    assert torch.equal(out_t, out_i)
    for r in range(len(c.lens)):
        assert torch.equal(c.pool.tensor[int(c.rs_np[r])], twin[int(c.ws_np[r])])
    assert gdn.get_device_error() == 0


@pytest.mark.slow
def test_chunked_long_sequence_close_to_exact(gdn):
    """32 chunks in one sequence (2048 tokens, 0.8B shape, bf16, twin):
    the chunked state and outputs stay within 1e-4 of the exact kernel's
    after every chunk boundary has carried the state on."""
    s = I.QWEN_08B
    c = Case(gdn, s, [2048, 77], seed=96, n_pad=0, token_slots=False)
    ref = c.prefill().clone()
    torch.cuda.synchronize()
    want = c.pool.tensor.cpu().numpy()
    c.reset()
    out = chunked(c)
    torch.cuda.synchronize()
    got = c.pool.tensor.cpu().numpy()
    for sl in c.ws_np:
        for h in range(s.hv):
            err = state_rel_err(got[sl, h], want[sl, h].astype(np.float64))
            assert err <= 1e-4, f"slot {sl} head {h}: {err:.3g}"
    assert_out_close(f64(out), f64(ref), "bf16")
    assert gdn.get_device_error() == 0


def test_chunked_graph_replay_equals_eager(gdn):
    """A captured gdn_prefill_chunked (twin) replays to the eager launch's
    outputs and states, bit for bit (the call enqueues only device work)."""
    s = I.QWEN_08B
    c = Case(gdn, s, [130, 64, 7], seed=97, n_pad=0, token_slots=False)
    out = torch.empty((c.T, s.hv, s.dv), dtype=torch.bfloat16, device="cuda")
    chunked(c, out=out)
    torch.cuda.synchronize()
    want_out, want_pool = out.clone(), c.pool.tensor.clone()
    c.reset()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            chunked(c, out=out)
    torch.cuda.current_stream().wait_stream(side)
    c.reset()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want_out)
    assert torch.equal(c.pool.tensor, want_pool)
    assert gdn.get_device_error() == 0


def test_chunked_decreasing_cu_seqlens_is_refused_per_sequence(gdn):
    """cu_seqlens that decreases (overlapping token ranges) cannot place every
    chunk in the prep workspace: cu = [0, 300, 0, 200] gives sequence 1 a
    negative range (bad) and sequence 2 the workspace units of sequence 0's
    chunks 2-4.  Sequence 0 still computes (its state and its tokens that no
    other sequence names match the exact kernel); sequence 2 is refused as a
    bad sequence: its state is untouched and the device error word is set."""
    s = I.QWEN_08B
    c = Case(gdn, s, [300, 0, 200], seed=98, n_pad=0, token_slots=False)
    cu = np.array([0, 300, 0, 200], dtype=np.int32)
    c.cu = ti(cu)
    ref_out = c.prefill().clone()   # the exact kernel on the same tables
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 1  # sequence 1's range
    ref_pool = c.pool.tensor.clone()
    c.reset()
    start = c.pool.tensor.clone()
    out = chunked(c)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 1
    ws0, ws2 = int(c.ws_np[0]), int(c.ws_np[2])
    got = c.pool.tensor.cpu().numpy()
    want = ref_pool.cpu().numpy()
    for h in range(s.hv):
        err = state_rel_err(got[ws0, h], want[ws0, h].astype(np.float64))
        assert err <= 5e-5, f"sequence 0 head {h}: {err:.3g}"
    assert torch.equal(c.pool.tensor[ws2], start[ws2])
    assert_out_close(f64(out[200:300]), f64(ref_out[200:300]), "bf16")


def test_chunked_output_not_16_byte_aligned(gdn):
    """The call does not require `out` to be 16-byte aligned: an output view
    2 bytes past an aligned buffer gets the same values as an aligned one
    (the kernel then stores its output rows 2 bytes at a time)."""
    c = Case(gdn, I.QWEN_08B, [130, 64, 1], seed=95, n_pad=0)
    T = int(c.cu_np[-1])
    n = T * c.s.hv * c.s.dv
    before = c.pool.tensor.clone()
    out_a = chunked(c, keep_in_place=False)
    torch.cuda.synchronize()
    after = c.pool.tensor.clone()
    c.pool.tensor.copy_(before)
    buf = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")
    view = buf[1:1 + n].view(T, c.s.hv, c.s.dv)
    assert view.data_ptr() % 16 == 2
    chunked(c, keep_in_place=False, out=view)
    torch.cuda.synchronize()
    assert torch.equal(view, out_a)
    assert torch.equal(c.pool.tensor, after)
    assert buf[0].item() == 0 and not buf[1 + n:].any()
    assert gdn.get_device_error() == 0


def test_chunked_ragged_tail_ignores_the_next_sequence(gdn):
    """A sequence's last, partial chunk is read by the tensor copies as a
    whole 64-token box, so its rows past the sequence hold the next
    sequence's tokens.  Those rows reach no result: with the next sequence's
    q, k and v all NaN, the first sequence's outputs and state are bit-equal
    to a run where they are ordinary values."""
    c = Case(gdn, I.QWEN_08B, [100, 80], seed=96, n_pad=0)
    a, b = int(c.cu_np[0]), int(c.cu_np[1])
    assert b - a == 100 and c.rs_np[0] > 0 and c.rs_np[1] > 0
    out_ok = chunked(c).clone()
    torch.cuda.synchronize()
    state_ok = c.pool.tensor[int(c.ws_np[0])].clone()
    c.reset()
    for k in ("q", "k", "v"):
        c.dev[k][b:] = float("nan")
    out_nan = chunked(c)
    torch.cuda.synchronize()
    assert torch.equal(out_nan[a:b], out_ok[a:b])
    assert torch.equal(c.pool.tensor[int(c.ws_np[0])], state_ok)
    assert torch.isnan(out_nan[b:].float()).any()  # the poisoned sequence itself is NaN
    assert gdn.get_device_error() == 0
