"""The calls inside a CUDA graph: captured once on preallocated buffers (outputs, status
words, workspaces), replayed on new inputs copied into the captured input buffers. Every
kernel is a programmatic dependent launch, so this checks those dependencies under
capture as well. And calls of every kind in flight at once on separate streams."""
import numpy as np
import pytest
import torch

from speculative_decoding_token_temp_gb300 import api, synth

from gpu_util import compare_greedy, compare_stochastic, handmade, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def test_stochastic_and_greedy_calls_replay_in_a_graph(dev):
    ws = [handmade(6, 4, 20000, synth.BF16, T=0.8, seed=120 + k) for k in range(3)]
    src = [dict(t=to_dev(w.target, dev), d=to_dev(w.draft, dev), tok=to_dev(w.tokens, dev),
                ua=to_dev(w.u_accept, dev), us=to_dev(w.u_sample, dev)) for w in ws]
    buf = {k: v.clone() for k, v in src[0].items()}
    s_out, g_out = {}, {}
    s_ws = torch.empty(8 << 20, dtype=torch.uint8, device=dev)
    g_ws = torch.empty(8 << 20, dtype=torch.uint8, device=dev)

    def calls():
        s_out["device_status"].zero_()
        g_out["device_status"].zero_()
        api.spec_verify_stochastic(buf["t"], buf["d"], buf["tok"], 0.8, buf["ua"], buf["us"], gamma=4, out=s_out,
                                   workspace=s_ws)
        api.spec_verify_greedy(buf["t"], buf["tok"], gamma=4, out=g_out, workspace=g_ws)

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        s_out["device_status"] = torch.zeros(1, dtype=torch.int32, device=dev)
        g_out["device_status"] = torch.zeros(1, dtype=torch.int32, device=dev)
        calls()                       # allocates every output once and sets kernel attributes
    torch.cuda.current_stream(dev).wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        calls()
    for k in (1, 2, 0):
        for name, v in src[k].items():
            buf[name].copy_(v)
        graph.replay()
        torch.cuda.synchronize()
        sr = {n: v.cpu().numpy() for n, v in s_out.items()}
        gr = {n: v.cpu().numpy() for n, v in g_out.items()}
        assert sr["device_status"][0] == 0 and gr["device_status"][0] == 0
        compare_stochastic(ws[k], sr, range(ws[k].B), T=0.8)
        compare_greedy(ws[k], gr, range(ws[k].B))


def test_multi_draft_replays_in_a_graph(dev):
    from test_gpu_multi import compare_multi
    G, K, gamma = 4, 3, 3
    ws = [synth.make_multi(G, K, gamma, 4096, synth.BF16, 0.8, seed=130 + k) for k in range(2)]
    src = [dict(t=to_dev(w.target, dev), d=to_dev(w.draft, dev), tok=to_dev(w.tokens, dev),
                ua=to_dev(w.u_accept, dev), us=to_dev(w.u_sample, dev)) for w in ws]
    buf = {k: v.clone() for k, v in src[0].items()}
    out = {}
    m_ws = torch.empty(8 << 20, dtype=torch.uint8, device=dev)

    def call():
        out["device_status"].zero_()
        api.spec_verify_multi(buf["t"], buf["d"], buf["tok"], K, 0.8, stochastic=True, u_accept=buf["ua"],
                              u_sample=buf["us"], out=out, workspace=m_ws)

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        out["device_status"] = torch.zeros(1, dtype=torch.int32, device=dev)
        call()
    torch.cuda.current_stream(dev).wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    for k in (1, 0):
        for name, v in src[k].items():
            buf[name].copy_(v)
        graph.replay()
        torch.cuda.synchronize()
        res = {n: v.cpu().numpy() for n, v in out.items()}
        assert res["device_status"][0] == 0
        compare_multi(ws[k], res, G, K, gamma, True)


def test_concurrent_calls_on_separate_streams(dev):
    """Calls of every kind in flight at once on four streams, each with its own workspace
    and outputs: a dense bf16 stochastic batch, a ragged fp32 stochastic batch, a greedy
    batch and a tree batch. The library keeps no state between calls outside the caller's
    buffers (device waves are looked up once per device), so every concurrent result equals
    the same call's result run alone; checked over five rounds, each also against the
    oracle once."""
    ws = [synth.make_stochastic(24, 50000, synth.BF16, 0.7, seed=91, gamma=6),
          synth.make_stochastic(17, 32003, synth.F32, 1.1, seed=92, gamma_range=(0, 9), agreement=0.6)]
    g = synth.make_stochastic(30, 40000, synth.BF16, 1.0, seed=93, gamma=5)
    tw = synth.make_tree(6, 60000, synth.BF16, seed=94)

    def inputs(w):
        cu = None if w.dense else torch.from_numpy(w.cu_draft).to(dev)
        gam = int(w.gammas[0]) if w.dense else w.gamma_max
        return dict(t=to_dev(w.target, dev), d=to_dev(w.draft, dev), tok=to_dev(w.tokens, dev),
                    ua=to_dev(w.u_accept, dev), us=to_dev(w.u_sample, dev), cu=cu, gam=gam)

    xs = [inputs(w) for w in ws]
    xg = inputs(g)
    tt, tn = to_dev(tw.target, dev), to_dev(tw.node_tokens, dev)

    def calls():
        outs = []
        for w, x in zip(ws, xs):
            outs.append(lambda w=w, x=x: api.spec_verify_stochastic(x["t"], x["d"], x["tok"], w.T, x["ua"], x["us"],
                                                                    cu_draft=x["cu"], gamma=x["gam"]))
        outs.append(lambda: api.spec_verify_greedy(xg["t"], xg["tok"], gamma=xg["gam"]))
        outs.append(lambda: api.spec_verify_tree(tt, tn, list(tw.parent)))
        return outs

    def host(res):
        return {k: v.cpu().numpy() for k, v in res.items() if k != "stats"}

    alone = []
    for fn in calls():
        r = fn()
        torch.cuda.synchronize()
        alone.append(host(r))
    for w, r in zip(ws, alone[:2]):
        assert int(r["device_status"][0]) == 0
        compare_stochastic(w, r, range(w.B))
    compare_greedy(g, alone[2], range(g.B))
    streams = [torch.cuda.Stream(dev) for _ in range(4)]
    for _ in range(5):
        res = []
        for s, fn in zip(streams, calls()):
            s.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(s):
                res.append(fn())
        torch.cuda.synchronize()
        for a, r in zip(alone, res):
            r = host(r)
            for k in a:
                assert np.array_equal(a[k], r[k], equal_nan=a[k].dtype.kind == "f"), k
