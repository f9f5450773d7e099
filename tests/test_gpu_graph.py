"""A Dion3 step captured in a CUDA graph and replayed gives bit-identical
results to the same steps enqueued eagerly: every call of the path enqueues
kernels only (no host synchronisation, no allocation), so it can be captured,
and a replay runs the same kernels on the same buffers."""
import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_shape_gb300 as d3
import workloads
from tests._harness import to_dev, to_host

pytestmark = pytest.mark.gpu

SHAPES = [(300, 200, 3, "bf16"), (96, 520, 2, "f32"), (1024, 1024, 2, "bf16")]


def _build(f, seed):
    groups, Ms, Ws, sels = [], [], [], []
    for gi, (n, m, batch, pd) in enumerate(SHAPES):
        M = [to_dev(workloads.gapped_momentum(n, m, seed=seed + 10 * gi + b)) for b in range(batch)]
        W = [to_dev(workloads.gaussian((n, m), 0.02, seed=seed + 100 + 10 * gi + b, dtype=pd), pd)
             for b in range(batch)]
        G = [to_dev(workloads.gaussian((n, m), 0.01, seed=seed + 200 + 10 * gi + b, dtype="bf16"), "bf16")
             for b in range(batch)]
        groups.append(d3.Group(params=W, grads=G, momentum=M))
        Ms.append(M)
        Ws.append(W)
        sels.append(torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda"))
    return groups, Ms, Ws, sels


@pytest.mark.parametrize("f", [0.25, 1.0])
def test_graph_replay_matches_eager(cuda_lib, f):
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)
    eager = _build(f, seed=11)
    graphed = _build(f, seed=11)
    ws_e = d3.alloc_workspace(d3.workspace_size(eager[0], hp))
    ws_g = d3.alloc_workspace(d3.workspace_size(graphed[0], hp))
    for _ in range(3):
        d3.step(eager[0], hp, ws_e, sel_idx_out=eager[3])
    torch.cuda.synchronize()
    d3.device_status()

    # Capture one step (the library's one-time set-up already ran above).
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        d3.step(graphed[0], hp, ws_g, sel_idx_out=graphed[3])   # current stream: the capturing one
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    d3.device_status()

    for gi in range(len(SHAPES)):
        assert np.array_equal(eager[3][gi].cpu().numpy(), graphed[3][gi].cpu().numpy())
        for a, b in zip(eager[1][gi], graphed[1][gi]):
            assert np.array_equal(to_host(a), to_host(b))
        for a, b in zip(eager[2][gi], graphed[2][gi]):
            assert np.array_equal(to_host(a), to_host(b))


def test_concurrent_groups_match_in_order(cuda_lib):
    """Several groups in one call, with the launch trace off and on (events
    between the launches, groups in order on the caller's stream): the groups
    share nothing, so both give bit-identical results."""
    f = 0.25
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)
    conc = _build(f, seed=23)
    seq = _build(f, seed=23)
    ws_c = d3.alloc_workspace(d3.workspace_size(conc[0], hp))
    ws_s = d3.alloc_workspace(d3.workspace_size(seq[0], hp))
    for _ in range(2):
        d3.step(conc[0], hp, ws_c, sel_idx_out=conc[3])
    d3.trace_enable(True)
    try:
        for _ in range(2):
            d3.step(seq[0], hp, ws_s, sel_idx_out=seq[3])
        torch.cuda.synchronize()
        trace = d3.trace_collect()
    finally:
        d3.trace_enable(False)
    assert sum(v["launches"] for v in trace.values()) > 0
    torch.cuda.synchronize()
    d3.device_status()
    for gi in range(len(SHAPES)):
        assert np.array_equal(conc[3][gi].cpu().numpy(), seq[3][gi].cpu().numpy())
        for a, b in zip(conc[1][gi] + conc[2][gi], seq[1][gi] + seq[2][gi]):
            assert np.array_equal(to_host(a), to_host(b))


def test_trace_counts_launches_and_work(cuda_lib):
    """The launch trace over one step: each Newton-Schulz run's 18 GEMMs
    (T = 5, restart before iteration 3) are timed as one chain but counted as
    18 launches, with the useful FLOPs 6 s^2 L + 14 s^3 per matrix; every
    memory-bound kernel launches once per group."""
    f = 0.25
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)
    groups, _, _, sels = _build(f, seed=31)
    ws = d3.alloc_workspace(d3.workspace_size(groups, hp))
    d3.step(groups, hp, ws, sel_idx_out=sels)
    d3.trace_enable(True)
    try:
        d3.step(groups, hp, ws, sel_idx_out=sels)
        trace = d3.trace_collect()
    finally:
        d3.trace_enable(False)
    d3.device_status()
    gemm = trace["gemm_tcgen05"]
    assert gemm["launches"] == 18 * len(SHAPES)
    want = 0.0
    for n, m, batch, _ in SHAPES:
        k = d3.num_selected(f, n)
        s, L = min(k, m), max(k, m)
        assert d3.useful_flops(k, m, hp) == pytest.approx(6.0 * s * s * L + 14.0 * s ** 3, rel=1e-12)
        want += d3.useful_flops(k, m, hp) * batch
    assert gemm["useful_flops"] == pytest.approx(want, rel=1e-9)
    assert gemm["total_ms"] > 0
    for name in ("topk_select", "gather_normalize"):
        assert trace[name]["launches"] == len(SHAPES), name
        assert trace[name]["total_ms"] > 0
    # Each group's accumulation: standalone, or (overlapped with the previous
    # group's Newton-Schulz GEMMs) a pool finished by one pool kernel.
    acc = sum(trace[n]["launches"] for n in ("accum_rownorm", "accum_pool") if n in trace)
    assert acc == len(SHAPES)
    # Each group's scatter update: its own launch, or (the two groups before
    # the last, whose rows all take the vector path here) rows of the scatter
    # pool carried by the last group's GEMM launches and finished by one pool
    # kernel.
    assert trace["scatter_update"]["launches"] == len(SHAPES) - 2
    assert trace["scatter_pool"]["launches"] == 1
    assert trace["scatter_pool"]["total_ms"] > 0


@pytest.mark.parametrize("lazy", [False, True])
def test_overlapped_groups_match_single_group_calls(cuda_lib, lazy):
    """One call over several groups (each group's accumulation overlapped with
    the previous group's Newton-Schulz GEMMs: rows taken by the GEMM launches'
    streaming warps and by the pool kernel) against the same groups stepped one
    call at a time (standalone accumulation): selections, momenta and
    parameters bit-identical over three steps."""
    f = 0.25
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)
    multi = _build(f, seed=41)
    single = _build(f, seed=41)
    scales = [[torch.ones((b, n), dtype=torch.float32, device="cuda") for (n, m, b, _) in SHAPES]
              for _ in range(2)]
    ws_m = d3.alloc_workspace(d3.workspace_size(multi[0], hp))
    ws_s = [d3.alloc_workspace(d3.workspace_size([g], hp)) for g in single[0]]
    for _ in range(3):
        if lazy:
            d3.step_lazy(multi[0], hp, scales[0], ws_m, sel_idx_out=multi[3])
        else:
            d3.step(multi[0], hp, ws_m, sel_idx_out=multi[3])
        for gi, g in enumerate(single[0]):
            if lazy:
                d3.step_lazy([g], hp, [scales[1][gi]], ws_s[gi], sel_idx_out=[single[3][gi]])
            else:
                d3.step([g], hp, ws_s[gi], sel_idx_out=[single[3][gi]])
    torch.cuda.synchronize()
    d3.device_status()
    for gi in range(len(SHAPES)):
        assert np.array_equal(multi[3][gi].cpu().numpy(), single[3][gi].cpu().numpy())
        for a, b in zip(multi[1][gi] + multi[2][gi], single[1][gi] + single[2][gi]):
            assert np.array_equal(to_host(a), to_host(b))
        assert np.array_equal(to_host(scales[0][gi]), to_host(scales[1][gi]))


def test_overlap_on_and_off_bitwise(cuda_lib):
    """dion3_set_overlap: the same three steps with the accumulation overlap
    off (groups on concurrent streams, standalone accumulation) and on give
    bit-identical selections, momenta and parameters."""
    f = 0.5
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)
    runs = []
    try:
        for on in (False, True):
            d3.set_overlap(on)
            st = _build(f, seed=53)
            ws = d3.alloc_workspace(d3.workspace_size(st[0], hp))
            for _ in range(3):
                d3.step(st[0], hp, ws, sel_idx_out=st[3])
            torch.cuda.synchronize()
            d3.device_status()
            runs.append(st)
    finally:
        d3.set_overlap(True)
    a, b = runs
    for gi in range(len(SHAPES)):
        assert np.array_equal(a[3][gi].cpu().numpy(), b[3][gi].cpu().numpy())
        for x, y in zip(a[1][gi] + a[2][gi], b[1][gi] + b[2][gi]):
            assert np.array_equal(to_host(x), to_host(y))


def test_overlap_with_groups_that_cannot_be_pooled(cuda_lib):
    """The overlapped schedule with groups whose accumulation cannot be a pool
    (130 matrices, more than a pool holds; 70 columns, not a multiple of 8):
    they accumulate with the standalone kernel in their turn.  Against the same
    groups stepped one call at a time: bit-identical over two steps."""
    shapes = [(64, 64, 130, "bf16"), (40, 70, 3, "f32"), (300, 200, 2, "bf16")]
    f = 0.5
    hp = d3.HParams(f=f, mu=0.9, lr=0.01)

    def build():
        groups, sels = [], []
        for gi, (n, m, batch, pd) in enumerate(shapes):
            M = [to_dev(workloads.gapped_momentum(n, m, seed=900 + 1000 * gi + b)) for b in range(batch)]
            W = [to_dev(workloads.gaussian((n, m), 0.02, seed=901 + 1000 * gi + b, dtype=pd), pd)
                 for b in range(batch)]
            G = [to_dev(workloads.gaussian((n, m), 0.01, seed=902 + 1000 * gi + b, dtype="bf16"), "bf16")
                 for b in range(batch)]
            groups.append(d3.Group(params=W, grads=G, momentum=M))
            sels.append(torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda"))
        return groups, sels

    multi, sel_m = build()
    single, sel_s = build()
    ws_m = d3.alloc_workspace(d3.workspace_size(multi, hp))
    ws_s = [d3.alloc_workspace(d3.workspace_size([g], hp)) for g in single]
    for _ in range(2):
        d3.step(multi, hp, ws_m, sel_idx_out=sel_m)
        for gi, g in enumerate(single):
            d3.step([g], hp, ws_s[gi], sel_idx_out=[sel_s[gi]])
    torch.cuda.synchronize()
    d3.device_status()
    for gi in range(len(shapes)):
        assert np.array_equal(sel_m[gi].cpu().numpy(), sel_s[gi].cpu().numpy())
        for a, b in zip(list(multi[gi].params) + list(multi[gi].momentum),
                        list(single[gi].params) + list(single[gi].momentum)):
            assert np.array_equal(to_host(a), to_host(b))


@pytest.mark.parametrize("ns_dtype", ["f16", "bf16"])
def test_deferred_scatter_with_more_groups_than_the_pool_holds(cuda_lib, ns_dtype):
    """Four groups: the last group's GEMM launches carry the scatter updates
    of the two groups before it (a scatter pool of two segments), the first
    group keeps its own scatter launch; O in fp16 or bf16, parameters in fp32
    and bf16 (the deferred pair is, in Newton-Schulz order, a bf16 and an fp32
    group).  Against the same groups stepped one call at a time:
    bit-identical selections, momenta and parameters over two steps, and the
    launch counts of that schedule."""
    shapes = [(256, 128, 4, "bf16"), (128, 256, 3, "bf16"), (96, 72, 5, "bf16"), (200, 136, 2, "f32")]
    f = 0.5
    hp = d3.HParams(f=f, mu=0.9, lr=0.01, ns_dtype=d3.BF16 if ns_dtype == "bf16" else d3.F16)

    def build():
        groups, sels = [], []
        for gi, (n, m, batch, pd) in enumerate(shapes):
            M = [to_dev(workloads.gapped_momentum(n, m, seed=700 + 1000 * gi + b)) for b in range(batch)]
            W = [to_dev(workloads.gaussian((n, m), 0.02, seed=701 + 1000 * gi + b, dtype=pd), pd)
                 for b in range(batch)]
            G = [to_dev(workloads.gaussian((n, m), 0.01, seed=702 + 1000 * gi + b, dtype="bf16"), "bf16")
                 for b in range(batch)]
            groups.append(d3.Group(params=W, grads=G, momentum=M))
            sels.append(torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda"))
        return groups, sels

    multi, sel_m = build()
    single, sel_s = build()
    ws_m = d3.alloc_workspace(d3.workspace_size(multi, hp))
    ws_s = [d3.alloc_workspace(d3.workspace_size([g], hp)) for g in single]
    d3.trace_enable(True)
    try:
        for _ in range(2):
            d3.step(multi, hp, ws_m, sel_idx_out=sel_m)
            trace = d3.trace_collect()
            for gi, g in enumerate(single):
                d3.step([g], hp, ws_s[gi], sel_idx_out=[sel_s[gi]])
            d3.trace_collect()
    finally:
        d3.trace_enable(False)
    torch.cuda.synchronize()
    d3.device_status()
    assert trace["scatter_update"]["launches"] == 2
    assert trace["scatter_pool"]["launches"] == 1
    for gi in range(len(shapes)):
        assert np.array_equal(sel_m[gi].cpu().numpy(), sel_s[gi].cpu().numpy())
        for a, b in zip(list(multi[gi].params) + list(multi[gi].momentum),
                        list(single[gi].params) + list(single[gi].momentum)):
            assert np.array_equal(to_host(a), to_host(b))


def test_deferred_scatter_carried_by_long_launches_bitwise(cuda_lib):
    """Groups of 8 to 32 matrices up to 2048 x 2048 at f = 1/2: the last
    group (32 matrices of 1024 x 2048, the least Newton-Schulz work) has
    rectangular and SYRK launches long enough for their streaming warps to
    take most of the deferred scatter rows of the two groups before it (the
    rest by the scatter pool kernel).  Two steps with the overlap on (deferred updates)
    and off (every group its own scatter launch) give bit-identical
    selections, momenta and parameters."""
    shapes = [(2048, 2048, 8, torch.bfloat16), (2048, 1024, 8, torch.float32), (1024, 2048, 32, torch.bfloat16)]
    f = 0.5
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)

    def build():
        groups, sels = [], []
        for gi, (n, m, batch, pd) in enumerate(shapes):
            M = [workloads.device_gaussian_(torch.empty((n, m), device="cuda"), 1.0, 5000 + 100 * gi + b)
                 for b in range(batch)]
            W = [workloads.device_gaussian_(torch.empty((n, m), device="cuda"), 0.02, 6000 + 100 * gi + b).to(pd)
                 for b in range(batch)]
            G = [workloads.device_gaussian_(torch.empty((n, m), device="cuda"), 0.01, 7000 + 100 * gi + b)
                 .to(torch.bfloat16) for b in range(batch)]
            groups.append(d3.Group(params=W, grads=G, momentum=M))
            sels.append(torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda"))
        return groups, sels

    runs = []
    try:
        for on in (True, False):
            d3.set_overlap(on)
            groups, sels = build()
            ws = d3.alloc_workspace(d3.workspace_size(groups, hp))
            for _ in range(2):
                d3.step(groups, hp, ws, sel_idx_out=sels)
            torch.cuda.synchronize()
            d3.device_status()
            runs.append((groups, sels))
    finally:
        d3.set_overlap(True)
    (ga, sa), (gb, sb) = runs
    for gi in range(len(shapes)):
        assert torch.equal(sa[gi], sb[gi])
        for x, y in zip(list(ga[gi].params) + list(ga[gi].momentum), list(gb[gi].params) + list(gb[gi].momentum)):
            assert torch.equal(x, y)


def test_all_zero_group_with_deferred_update_leaves_parameters_unchanged(cuda_lib):
    """A group whose momentum and gradients are all zero, stepped with two
    other groups: its update is deferred into the last group's launches (it
    has the most Newton-Schulz work, so it runs first), X = 0 / (0 + eps) and
    O are zero, and W - lr O leaves every parameter bit-identical; the
    momentum stays zero and the other groups match single-group calls."""
    shapes = [(512, 512, 4, "bf16"), (256, 384, 3, "f32"), (128, 256, 2, "bf16")]
    f = 0.5
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)

    def build(zero):
        groups, sels = [], []
        for gi, (n, m, batch, pd) in enumerate(shapes):
            if gi == 0 and zero:
                M = [torch.zeros((n, m), device="cuda") for _ in range(batch)]
                G = [torch.zeros((n, m), device="cuda", dtype=torch.bfloat16) for _ in range(batch)]
            else:
                M = [to_dev(workloads.gapped_momentum(n, m, seed=300 + 10 * gi + b)) for b in range(batch)]
                G = [to_dev(workloads.gaussian((n, m), 0.01, seed=301 + 10 * gi + b, dtype="bf16"), "bf16")
                     for b in range(batch)]
            W = [to_dev(workloads.gaussian((n, m), 0.02, seed=302 + 10 * gi + b, dtype=pd), pd) for b in range(batch)]
            groups.append(d3.Group(params=W, grads=G, momentum=M))
            sels.append(torch.empty((batch, d3.num_selected(f, n)), dtype=torch.int32, device="cuda"))
        return groups, sels

    multi, sel_m = build(True)
    w0 = [w.clone() for w in multi[0].params]
    single, sel_s = build(True)
    ws_m = d3.alloc_workspace(d3.workspace_size(multi, hp))
    ws_s = [d3.alloc_workspace(d3.workspace_size([g], hp)) for g in single]
    d3.trace_enable(True)
    try:
        d3.step(multi, hp, ws_m, sel_idx_out=sel_m)
        trace = d3.trace_collect()
    finally:
        d3.trace_enable(False)
    for gi, g in enumerate(single):
        d3.step([g], hp, ws_s[gi], sel_idx_out=[sel_s[gi]])
    torch.cuda.synchronize()
    d3.device_status()
    assert trace["scatter_pool"]["launches"] == 1
    for a, b in zip(multi[0].params, w0):
        assert torch.equal(a, b)
    for m in multi[0].momentum:
        assert not torch.any(m)
    for gi in range(1, len(shapes)):
        assert np.array_equal(sel_m[gi].cpu().numpy(), sel_s[gi].cpu().numpy())
        for a, b in zip(list(multi[gi].params) + list(multi[gi].momentum),
                        list(single[gi].params) + list(single[gi].momentum)):
            assert np.array_equal(to_host(a), to_host(b))


def test_normuon_with_deferred_updates_overlap_on_and_off_bitwise(cuda_lib):
    """dion3_step_normuon over three groups: with the overlap on, the two
    groups before the last have their normalised updates (each row's lr times
    its factor) carried by the last group's launches; with it off every group
    scatters on its own.  Two steps give bit-identical selections, momenta,
    parameters and second-moment states."""
    f = 0.5
    hp = d3.HParams(f=f, mu=0.95, lr=0.02)
    nm = d3.NormuonParams()
    runs = []
    try:
        for on in (True, False):
            d3.set_overlap(on)
            st = _build(f, seed=71)
            v = [torch.zeros((b, n), dtype=torch.float32, device="cuda") for (n, m, b, _) in SHAPES]
            ws = d3.alloc_workspace(d3.workspace_size(st[0], hp))
            for _ in range(2):
                d3.step_normuon(st[0], hp, nm, v, ws, sel_idx_out=st[3])
            torch.cuda.synchronize()
            d3.device_status()
            runs.append((st, v))
    finally:
        d3.set_overlap(True)
    (a, va), (b, vb) = runs
    for gi in range(len(SHAPES)):
        assert np.array_equal(a[3][gi].cpu().numpy(), b[3][gi].cpu().numpy())
        for x, y in zip(a[1][gi] + a[2][gi], b[1][gi] + b[2][gi]):
            assert np.array_equal(to_host(x), to_host(y))
        assert torch.equal(va[gi], vb[gi])
