"""moe_route_noalloc: routing for callers that cannot allocate device memory.

A caller whose device memory is all held by its own pool allocator, or whose
decode loop must not take cudaMalloc's implicit synchronisation, routes with
moe_route_noalloc into buffers it owns; the call's only scratch is a built-in
device array.  These tests call it through the C ABI and check, on two calls in
a row (the array keeps the previous call's contents), that it returns what
moe_route returns for the same inputs, that batches of more than 8 tokens
(which no layer call routes with a partial map) give the oracle's routing and
compaction bit for bit, and that sizes beyond the built-in array are refused
with a clear error.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from expert_offload_moe_gb300 import build as moe_build  # noqa: E402
from expert_offload_moe_gb300 import moe, stack, synth  # noqa: E402

from parity import W_ATOL, W_RTOL, compare_routing, route_arrays  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe_build.build()
    moe.lib()


def new_buffers(M, k, E):
    n = M * k
    i32 = dict(dtype=torch.int32, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    b = {name: torch.full((n,), -7, **i32) for name in
         ("topk_ids", "hot_expert", "hot_token", "act_expert", "act_slot", "act_off", "act_cnt",
          "cold_token", "cold_expert")}
    for name in ("topk_w", "hot_w", "cold_w"):
        b[name] = torch.full((n,), -7.0, **f32)
    b["hist"] = torch.full((E,), -7, **i32)
    b["counts"] = torch.full((4,), -7, **i32)
    return b


def check_same(bufs, ref, E, k):
    counts = bufs["counts"].cpu().numpy()
    assert np.array_equal(counts, ref["counts"])
    n_hot, n_cold, n_act, M = (int(c) for c in counts)
    got = {name: t.cpu().numpy() for name, t in bufs.items()}
    assert np.array_equal(got["topk_ids"][:M * k].reshape(M, k), ref["ids"])
    assert np.allclose(got["topk_w"][:M * k].reshape(M, k), ref["w"], rtol=W_RTOL, atol=W_ATOL)
    for name in ("hot_expert", "hot_token"):
        assert np.array_equal(got[name][:n_hot], ref[name])
    assert np.allclose(got["hot_w"][:n_hot], ref["hot_w"], rtol=W_RTOL, atol=W_ATOL)
    for name in ("act_expert", "act_slot", "act_off", "act_cnt"):
        assert np.array_equal(got[name][:n_act], ref[name])
    for name in ("cold_token", "cold_expert"):
        assert np.array_equal(got[name][:n_cold], ref[name])
    assert np.allclose(got["cold_w"][:n_cold], ref["cold_w"], rtol=W_RTOL, atol=W_ATOL)
    assert np.array_equal(got["hist"], ref["hist"])


@pytest.mark.parametrize("name,placement", [("tiny_h256_i128_e16k2", "partial"),
                                            ("e512k10_h2048_i512_s256_m1", "rank")])
def test_noalloc_route_matches_moe_route_twice_in_a_row(name, placement):
    w = synth.WORKLOADS[name]
    E, k, H = w.experts, w.top_k, w.hidden
    if placement == "partial":
        e2s = np.full(E, -1, dtype=np.int32)
        e2s[::2] = np.arange(len(e2s[::2]))
        w = synth.Workload(w.name + "_half", 1, H, w.inter, E, k, len(e2s[::2]), w.tokens, 1)
        li = stack.LayerInputs(w, 0, e2s=e2s)
    else:
        li = stack.LayerInputs(w, 2)
    lay = li.make_layer(max_tokens=8)
    Wr = torch.from_numpy(li.Wr).cuda()
    bias = torch.from_numpy(li.bias).cuda()
    e2s_dev = torch.from_numpy(np.ascontiguousarray(li.e2s, dtype=np.int32)).cuda()
    for call, M in enumerate((8, 3)):  # two calls in a row, different sizes and inputs
        x = stack.bf16_tensor(synth.activations(0, li.layer, 900 + call, M, H))
        ref = route_arrays(lay.route(x, M), E, k)
        bufs = new_buffers(M, k, E)
        moe.route_noalloc(x, M, Wr, bias, E, k, e2s_dev, bufs)
        torch.cuda.synchronize()
        check_same(bufs, ref, E, k)
    lay.close()


def read_buffers(bufs, k, E):
    counts = bufs["counts"].cpu().numpy()
    n_hot, n_cold, n_act, M = (int(c) for c in counts)
    h = {name: t.cpu().numpy() for name, t in bufs.items()}
    return {"counts": counts, "ids": h["topk_ids"][:M * k].reshape(M, k), "w": h["topk_w"][:M * k].reshape(M, k),
            "hot_expert": h["hot_expert"][:n_hot], "hot_token": h["hot_token"][:n_hot], "hot_w": h["hot_w"][:n_hot],
            "act_expert": h["act_expert"][:n_act], "act_slot": h["act_slot"][:n_act],
            "act_off": h["act_off"][:n_act], "act_cnt": h["act_cnt"][:n_act],
            "cold_token": h["cold_token"][:n_cold], "cold_expert": h["cold_expert"][:n_cold],
            "cold_w": h["cold_w"][:n_cold], "hist": h["hist"]}


@pytest.mark.parametrize("E,k,H,Ms,tau", [(16, 2, 256, (16, 600), 0.0), (512, 10, 2048, (16, 40), 0.25),
                                          (64, 10, 256, (128, 9), 0.0)])
def test_noalloc_route_batches_above_eight_tokens_match_the_oracle(E, k, H, Ms, tau):
    """Batches of more than 8 tokens take the route kernel's general compaction (route lists kept in
    global memory once M * k > 1024), which no layer call reaches with a partial map: top-k ids,
    hot / active / cold lists and counts must equal the oracle's bit for bit (near-tie tokens aside),
    with half the experts cold, on two calls in a row."""
    import oracle

    Wr_h = synth.router_weights(5, 1, E, H)
    b_h = synth.router_bias(5, 1, E, tau)
    e2s = np.full(E, -1, dtype=np.int32)
    e2s[1::2] = np.random.default_rng(E).permutation(E // 2)  # odd experts in shuffled slots
    Wr = torch.from_numpy(Wr_h).cuda()
    bias = torch.from_numpy(b_h).cuda()
    e2s_dev = torch.from_numpy(e2s).cuda()
    for call, M in enumerate(Ms):
        xb = synth.activations(5, 1, 300 + call, M, H)
        bufs = new_buffers(M, k, E)
        moe.route_noalloc(stack.bf16_tensor(xb), M, Wr, bias, E, k, e2s_dev, bufs)
        torch.cuda.synchronize()
        g = read_buffers(bufs, k, E)
        logits = oracle.router_logits(xb, Wr_h, b_h)
        ids, w = oracle.topk_softmax(logits, k)
        o = oracle.compact(ids, w, e2s)
        o.update(ids=ids, w=w)
        assert int(g["counts"][3]) == M
        excluded = compare_routing(g, o, logits, k, e2s)
        assert len(excluded) <= max(1, M // 50)
        assert g["counts"][0] > 0 and g["counts"][1] > 0  # both hot and cold routes were exercised


def test_noalloc_route_refuses_sizes_beyond_its_scratch():
    E, k, H, M = 512, 10, 2048, 128  # ceil(2048/256) * 128 * 512 * 4 bytes = 2 MiB > 1 MiB
    x = torch.zeros((M, H), dtype=torch.bfloat16, device="cuda")
    Wr = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    e2s = torch.arange(E, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.route_noalloc(x, M, Wr, None, E, k, e2s, new_buffers(M, k, E))
    assert ei.value.code == moe.MOE_EINVAL and "scratch" in str(ei.value)
