"""GPU parity: grouped SwiGLU FFN + combine against the oracle's float64
Eq. (1), on the same (oracle) routing.  Bar: max|dy| <= 2e-2 * rms(y_ref)."""
import numpy as np
import pytest
import torch

import oracle
import expert_routing_moe_gb300 as moe
from expert_routing_moe_gb300 import _abi as abi
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import _gpu
    return _gpu


@pytest.fixture(scope="module")
def qwen(g):
    """The Qwen3-30B-A3B-shaped decode layer (1.2 GB of bf16 experts), on the device once."""
    L = syn.decode(32)
    return L, g.DevLayer(L)


def _route(L, x_np, T, R=None, sere=False, protect=None, kp=2):
    xd = oracle.DT_BF16 if L.dtype == "bf16" else oracle.DT_F32
    l = oracle.router(x_np, L.w_r, xd)
    ids, gates = oracle.route(l, R or L.k)
    if sere:
        ids, gates, _, _ = oracle.sere(ids[:, :L.k], gates[:, :L.k], L.N, L.k, kp, 0.5, L.sim, protect)
    return ids[:, :L.k].copy(), gates[:, :L.k].copy()


def _ffn_case(g, L, D, x_np, x_dev, ids, gates, tokens=None, fuse=True):
    d = g.gpu_dispatch(g.dev(ids), g.dev(gates), L.N, L.k, L.k)
    y = g.gpu_ffn(x_dev, D.w_gate, D.w_up, D.w_down, L.k, d["dev"], x_dev.shape[0], fuse=fuse)
    xd = oracle.DT_BF16 if L.dtype == "bf16" else oracle.DT_F32
    wd = oracle.DT_BF16 if L.dtype == "bf16" else oracle.DT_F32
    yref = oracle.ffn_combine(x_np, L.w_gate, L.w_up, L.w_down, ids, gates, L.k, tokens, xd, wd)
    ysel = y if tokens is None else y[tokens]
    return g.assert_y_close(ysel, yref, "ffn")


def test_tiny_fp32(g):
    L = syn.tiny()
    D = g.DevLayer(L)
    ids, gates = _route(L, L.x, L.T)
    _ffn_case(g, L, D, L.x, D.x, ids, gates)
    _ffn_case(g, L, D, L.x, D.x, ids, gates, fuse=False)


@pytest.mark.parametrize("T", [1, 16, 32])
def test_decode_bf16(g, qwen, T):
    L, D = qwen
    Lt = syn.decode(T, with_weights=False, token_stream_offset=T)
    x_dev = g.dev(Lt.x_bf16, torch.bfloat16)
    ids, gates = _route(L, Lt.x_bf16, T)
    _ffn_case(g, L, D, Lt.x_bf16, x_dev, ids, gates)


def test_decode_bf16_sere_rows_out_and_combine(g, qwen):
    L, D = qwen
    ids, gates = _route(L, L.x_bf16, L.T, sere=True)
    assert (ids < 0).any()  # merged slots leave holes
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates, fuse=False)


def test_decode_bf16_batch128_sampled(g, qwen):
    L, D = qwen
    Lt = syn.sweep(128, with_weights=False)
    x_dev = g.dev(Lt.x_bf16, torch.bfloat16)
    ids, gates = _route(L, Lt.x_bf16, 128)
    tokens = np.arange(0, 128, 5, dtype=np.int32)
    _ffn_case(g, L, D, Lt.x_bf16, x_dev, ids, gates, tokens)


def test_small_bf16_multi_chunk_ragged(g):
    """T=200 (the weight-major kernel) with a skewed routing: the hottest
    expert has > 64 rows, so it is split into several token chunks with a
    ragged tail; H and I span several tiles."""
    L = syn.qwen_layer(200, H=384, N=16, k=4, I=256)
    D = g.DevLayer(L)
    rng = np.random.default_rng(0)
    ids = np.stack([np.concatenate([[0], rng.choice(np.arange(1, 16), 3, replace=False)]) for _ in range(200)])
    ids = ids.astype(np.int32)
    gates = rng.random((200, 4)).astype(np.float32)
    ids[rng.random(ids.shape) < 0.1] = -1
    gates[ids < 0] = 0
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates)


def test_small_bf16_odd_slice_count(g):
    """The decode kernel at I = 384 (six half-slice phase-1 units per expert)
    and H = 256 (two down-projection tiles)."""
    L = syn.qwen_layer(24, H=256, N=8, k=3, I=384)
    D = g.DevLayer(L)
    ids, gates = _route(L, L.x_bf16, 24)
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates)


def test_repeat_calls_are_stable(g, qwen):
    L, D = qwen
    ids, gates = _route(L, L.x_bf16, L.T)
    d = g.gpu_dispatch(g.dev(ids), g.dev(gates), L.N, L.k, L.k)
    ys = [g.gpu_ffn(D.x, D.w_gate, D.w_up, D.w_down, L.k, d["dev"], L.T) for _ in range(3)]
    yref = oracle.ffn_combine(L.x_bf16, L.w_gate, L.w_up, L.w_down, ids, gates, L.k, None, oracle.DT_BF16,
                              oracle.DT_BF16)
    for y in ys:
        g.assert_y_close(y, yref, "repeat")
    # fp32 atomics reorder sums only: repeated results agree far inside the bar
    assert np.max(np.abs(ys[0] - ys[1])) <= 1e-4 * np.sqrt(np.mean(yref ** 2))


def test_one_workspace_across_calls(g, qwen):
    """The weight-major kernel leaves its counters at zero: calls that share
    one workspace (zeroed once) agree with the oracle, across batch sizes
    that use different unit splits, and the counter words are zero after
    every call."""
    L, D = qwen
    ws = g.ffn_workspace(D.x, D.w_gate, L.k, L.T)
    for T in (L.T, 1, 5, L.T, 3):
        ids, gates = _route(L, L.x_bf16[:T], T)
        d = g.gpu_dispatch(g.dev(ids), g.dev(gates), L.N, L.k, L.k)
        for fuse in (True, False):
            y = g.gpu_ffn(D.x[:T], D.w_gate, D.w_up, D.w_down, L.k, d["dev"], T, fuse=fuse, ws=ws)
            yref = oracle.ffn_combine(L.x_bf16[:T], L.w_gate, L.w_up, L.w_down, ids, gates, L.k, None,
                                      oracle.DT_BF16, oracle.DT_BF16)
            g.assert_y_close(y, yref, "shared workspace T=%d fuse=%d" % (T, fuse))
            # the counter region: a fixed 2304 bytes at the start of the workspace
            assert int(ws[:2304].view(torch.int32).abs().sum().item()) == 0


def _skewed_ids(rng, T, N, k, hot=0, hole_frac=0.1):
    """Every token routes to expert `hot` plus k-1 others: `hot` gets T rows
    (many 128-row chunks and a ragged tail), the rest a few dozen each."""
    ids = np.stack([np.concatenate([[hot], rng.choice(np.delete(np.arange(N), hot), k - 1, replace=False)])
                    for _ in range(T)]).astype(np.int32)
    gates = rng.random((T, k)).astype(np.float32)
    ids[rng.random(ids.shape) < hole_frac] = -1
    gates[ids < 0] = 0
    return ids, gates


@pytest.mark.parametrize("fuse", [True, False])
def test_token_major_multi_chunk_ragged(g, fuse):
    """T = 1100 runs the token-major (prefill) kernel: expert 0 holds ~990
    rows (eight 128-row chunks, the last one ragged), the other experts hold
    one partial chunk each; H spans two 256-row down-projection tiles."""
    L = syn.qwen_layer(1100, H=512, N=8, k=2, I=256)
    D = g.DevLayer(L)
    ids, gates = _skewed_ids(np.random.default_rng(3), 1100, 8, 2)
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates, fuse=fuse)


@pytest.mark.parametrize("fuse", [True, False])
def test_token_major_item_boundaries(g, fuse):
    """Experts with 256, 128, 129, 1, 384, 97, 29 and 0 rows (k = 1, 1024
    tokens in shuffled order) in the token-major kernel's 128-row items:
    whole items, an expert of exactly one item, items followed by a
    single-row one, partial items and an empty expert."""
    counts = [256, 128, 129, 1, 384, 97, 29, 0]
    T = sum(counts)
    L = syn.qwen_layer(T, H=512, N=len(counts), k=1, I=256)
    D = g.DevLayer(L)
    rng = np.random.default_rng(5)
    ids = rng.permutation(np.repeat(np.arange(len(counts)), counts)).astype(np.int32)[:, None]
    gates = rng.random((T, 1)).astype(np.float32) + 0.25
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates, fuse=fuse)


def test_token_major_odd_tiles(g):
    """I = 384 (three slices) and H = 768 (three 256-row tiles) in the token-major kernel."""
    L = syn.qwen_layer(1024, H=768, N=6, k=3, I=384)
    D = g.DevLayer(L)
    ids, gates = _route(L, L.x_bf16, 1024)
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates)


@pytest.mark.parametrize("fuse", [True, False])
def test_token_major_many_ranks(g, fuse):
    """k = 12 > 8 in the token-major kernel: the combine's instance for up to
    16 rows per token (fused), or the rows added into the caller's buffer."""
    L = syn.qwen_layer(1024, H=256, N=32, k=12, I=128)
    D = g.DevLayer(L)
    ids, gates = _route(L, L.x_bf16, 1024)
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates, fuse=fuse)


@pytest.mark.parametrize("T,N,k,H,I", [
    (12, 64, 12, 256, 128),    # 16-column token tile, k = 12, two half units per expert
    (16, 128, 8, 256, 768),    # 16-column tile, full Qwen expert width
    (24, 64, 12, 256, 256),    # 32-column tile, 288 dispatch rows
    (30, 64, 16, 256, 256),    # 32-column tile, k = 16: 480 dispatch rows
])
def test_decode_kernel_odd_shapes(g, T, N, k, H, I):
    """The decode kernel (every batch of up to 64 tokens) at shapes off the
    Qwen one: k = 12 and 16, I = 128 and 256, H = 256; fused combine and
    rows out."""
    L = syn.qwen_layer(T, H=H, N=N, k=k, I=I)
    D = g.DevLayer(L)
    ids, gates = _route(L, L.x_bf16, T)
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates)
    _ffn_case(g, L, D, L.x_bf16, D.x, ids, gates, fuse=False)


def test_decode_kernel_max_experts(g):
    """N = 256 experts (the library's maximum) with k = 16 at a batch of 40:
    up to 256 active experts in the decode kernel's expert lists.  N(0, 1)
    activations, as in the weight-major shapes below (the synthetic x is
    scaled to rms ~300 at this shape)."""
    L = syn.qwen_layer(40, H=256, N=256, k=16, I=128)
    D = g.DevLayer(L)
    x_bits = syn.f32_to_bf16_bits(np.random.default_rng(40).standard_normal((40, 256)).astype(np.float32))
    x_dev = g.dev(x_bits, torch.bfloat16)
    ids, gates = _route(L, x_bits, 40)
    assert len(np.unique(ids[ids >= 0])) > 128
    _ffn_case(g, L, D, x_bits, x_dev, ids, gates)


@pytest.mark.parametrize("T,N,k,H,I", [
    (65, 64, 8, 256, 128),     # the smallest weight-major batch; one I-slice per expert
    (100, 128, 8, 256, 768),   # the Qwen expert width
    (300, 64, 12, 512, 256),   # k = 12: about 56 rows per expert, some in two 64-row chunks
    (80, 256, 16, 256, 128),   # N = 256 and k = 16: 255 active experts in the item table
    (1000, 32, 4, 256, 384),   # near the largest weight-major batch: two or three chunks per expert
])
def test_weight_major_kernel_shapes(g, T, N, k, H, I):
    """The weight-major kernel (batches of 65 to 1023 tokens: the weights as
    the 128-row MMA operand, each expert's rows in chunks of 64 as N), fused
    combine and rows out.  The activations are N(0, 1): the synthetic layers
    scale x to give their router logits a set spread, which at H = 256 means
    x of rms ~400 and a y whose largest elements are 13x its rms, where the
    bf16 rounding of the SwiGLU activations alone reaches 2e-2 * rms."""
    L = syn.qwen_layer(T, H=H, N=N, k=k, I=I)
    D = g.DevLayer(L)
    x_bits = syn.f32_to_bf16_bits(np.random.default_rng(T).standard_normal((T, H)).astype(np.float32))
    x_dev = g.dev(x_bits, torch.bfloat16)
    ids, gates = _route(L, x_bits, T)
    _ffn_case(g, L, D, x_bits, x_dev, ids, gates)
    _ffn_case(g, L, D, x_bits, x_dev, ids, gates, fuse=False)


def test_token_major_prefill_shape_sampled(g, qwen):
    """The prefill shape (T = 8192, H = 2048, I = 768, 128 experts, top-8) on
    plain top-8 routing; sampled tokens against the oracle."""
    L, D = qwen
    Lt = syn.prefill(with_weights=False)
    x_dev = g.dev(Lt.x_bf16, torch.bfloat16)
    ids, gates = _route(L, Lt.x_bf16, Lt.T)
    tokens = np.sort(np.random.default_rng(11).choice(Lt.T, 1024, replace=False)).astype(np.int32)
    oracle.set_threads(0)
    _ffn_case(g, L, D, Lt.x_bf16, x_dev, ids, gates, tokens)


@pytest.mark.parametrize("fuse", [True, False])
def test_token_major_shared_workspace_and_empty_dispatch(g, fuse):
    """Three token-major calls on one workspace (zeroed once): a normal batch,
    a batch whose every slot is empty (no units at all: y must still be
    written, as zeros), the normal batch again; each matches the oracle."""
    L = syn.qwen_layer(1100, H=512, N=8, k=2, I=256)
    D = g.DevLayer(L)
    ids, gates = _skewed_ids(np.random.default_rng(5), 1100, 8, 2)
    empty_ids = np.full_like(ids, -1)
    empty_gates = np.zeros_like(gates)
    ws = g.ffn_workspace(D.x, D.w_gate, L.k, L.T)
    for ii, gg in ((ids, gates), (empty_ids, empty_gates), (ids, gates)):
        d = g.gpu_dispatch(g.dev(ii), g.dev(gg), L.N, L.k, L.k)
        y = g.gpu_ffn(D.x, D.w_gate, D.w_up, D.w_down, L.k, d["dev"], L.T, fuse=fuse, ws=ws)
        if (ii < 0).all():
            assert np.all(y == 0.0)
        else:
            yref = oracle.ffn_combine(L.x_bf16, L.w_gate, L.w_up, L.w_down, ii, gg, L.k, None, oracle.DT_BF16,
                                      oracle.DT_BF16)
            g.assert_y_close(y, yref, "token-major shared workspace fuse=%d" % fuse)


def test_dependency_wait_times_out_cleanly(g, qwen):
    """Failure detection without a fault: the work counter is preset past the
    phase-1 units, so after its static first unit every CTA draws only
    phase-2 units, and the experts whose phase-1 units were skipped never
    publish their activations (a flag that nothing sets).  The bounded wait runs
    out, the launch reports MOE_DEV_TIMEOUT at the dependency site and
    returns; the last CTA still returns the counters to zero, so the same
    workspace then serves a normal call."""
    L, D = qwen
    ids, gates = _route(L, L.x_bf16, L.T)
    d = g.gpu_dispatch(g.dev(ids), g.dev(gates), L.N, L.k, L.k)
    ws = g.ffn_workspace(D.x, D.w_gate, L.k, L.T)
    # batch 32: one 32-row chunk per active expert and I / 64 phase-1 units
    # each (half slices: 64 gate and 64 up rows stacked)
    n1 = int(d["active"][0]) * (L.I // 64)
    ws[:4].view(torch.int32)[0] = n1
    y = torch.full((L.T, L.H), float("nan"), dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_ffn_grouped(D.x, D.w_gate, D.w_up, D.w_down, L.k, d["dev"]["offsets"], d["dev"]["row_token"],
                        d["dev"]["row_gate"], d["dev"]["active"], y, ws, abi.MOE_FFN_FUSE_COMBINE | abi.MOE_FFN_ZERO_Y,
                        st)
    torch.cuda.synchronize()
    code, detail = (int(v) for v in st.tolist())
    assert code == abi.MOE_DEV_TIMEOUT, (code, detail)
    # the dependency wait, or a wait of another warp role on the same missing data
    # (the first one to give up reports its site)
    assert 1 <= detail <= 10, detail
    assert int(ws[:2304].view(torch.int32).abs().sum().item()) == 0
    # the context and the workspace are usable again
    y2 = g.gpu_ffn(D.x, D.w_gate, D.w_up, D.w_down, L.k, d["dev"], L.T, ws=ws)
    yref = oracle.ffn_combine(L.x_bf16, L.w_gate, L.w_up, L.w_down, ids, gates, L.k, None, oracle.DT_BF16,
                              oracle.DT_BF16)
    g.assert_y_close(y2, yref, "after a timed-out call")
