"""The row-sharded LM head (small-vocabulary MTP study, section 3.3: verify against the full
vocabulary) split over ranks.

CPU, no GPU: the oracle's slice winners and their merge against the whole-head argmax (pins),
the slice plan, and two gloo ranks running the protocol end to end -- each rank scores its
slice with the oracle, the ranks all-gather their winners with the library's gather step, and
both ranks must reach the whole-head oracle's argmax and acceptance; and two gloo ranks running
lmhead_verify_sharded itself with host stand-ins for its two kernels (score, gather, merge in
that order, each rank's keys at its own row of the gathered array).
GPU: slices scored by lmhead_argmax_partial on one GPU, merged by lmhead_accept_keys, against
the oracle (the all-gather is then a concatenation on one device; the kernels never wait on one
another)."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

import synth
from oracle import int4 as oint4
from oracle import verify as over

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_shard_rows_cover_the_head_once():
    from bit_weight_gemv_gb300.sharded import shard_rows
    for N in (8, 9, 1000, 248_320):
        for W in (1, 2, 3, 4, 8):
            rows = []
            for r in range(W):
                off, n = shard_rows(N, W, r)
                rows.extend(range(off, off + n))
                assert n in (N // W, N // W + 1)
            assert rows == list(range(N))
    with pytest.raises(ValueError):
        shard_rows(3, 4, 0)


def test_merge_of_slice_winners_is_the_whole_head_argmax():
    g = np.random.default_rng(7)
    for trial in range(200):
        M, N = 5, int(g.integers(4, 40))
        logits = g.integers(-3, 4, size=(M, N)).astype(np.float64)  # many exact ties
        W = int(g.integers(1, min(N, 6) + 1))
        cuts = np.sort(g.choice(np.arange(1, N), size=W - 1, replace=False)) if W > 1 else []
        bounds = [0, *cuts, N]
        vals, rows = [], []
        order = g.permutation(W)  # shard order in the gathered array is free
        for w in order:
            v, r = over.shard_winners(logits[:, bounds[w]:bounds[w + 1]], bounds[w])
            vals.append(v)
            rows.append(r)
        assert np.array_equal(over.merge_winners(np.array(vals), np.array(rows)),
                              over.argmax_lowest(logits)), trial


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import synth as sy
        from oracle import int4 as oi
        from oracle import verify as ov
        from bit_weight_gemv_gb300.sharded import gather_keys, shard_rows
        M, N, K = 16, 1001, 256
        codes, scales, h = sy.int4_problem(51, M, N, K)        # the same head on every rank
        off, n = shard_rows(N, world, rank)
        v, r = ov.shard_winners(oi.gemm(h, codes[off:off + n], scales[off:off + n]), off)
        vals = torch.empty((world, M), dtype=torch.float64)
        rows = torch.empty((world, M), dtype=torch.int64)
        gather_keys(torch.from_numpy(v), vals)
        gather_keys(torch.from_numpy(r.astype(np.int64)), rows)
        a = ov.merge_winners(vals.numpy(), rows.numpy())
        full = ov.argmax_lowest(oi.gemm(h, codes, scales))
        drafts, j = sy.plant_drafts(52, full, N, 6)
        q.put((rank, a.tolist(), full.tolist(), ov.accept(a, drafts), j))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reach_the_whole_head_result():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, a, full, (n, b), j in got:
        assert a == full
        assert n == j and b == full[n]
    assert got[0][1] == got[1][1]


def _key(value, row):
    """The slice key of the library (reading 17): order-preserving fp32 bits of the logit above
    0xFFFFFFFF - global row, so the largest key is the largest logit, then the lowest row."""
    b = int(np.float32(value).view(np.uint32))
    ordered = (b ^ 0xFFFFFFFF) if b & 0x80000000 else (b | 0x80000000)
    return (ordered << 32) | (0xFFFFFFFF - int(row))  # unsigned 64-bit


def _rank_flow(rank, world, port, q):
    """One rank of lmhead_verify_sharded with the two kernels replaced by host stand-ins (the
    oracle's slice scores packed into keys; the merge of the gathered keys), so the host
    sequence -- score, all-gather, merge -- runs over gloo without a GPU."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import synth as sy
        from oracle import int4 as oi
        from oracle import verify as ov
        import bit_weight_gemv_gb300 as lb
        from bit_weight_gemv_gb300.sharded import lmhead_verify_sharded, shard_rows
        M, N, K = 16, 1001, 256
        codes, scales, h = sy.int4_problem(53, M, N, K)
        full = ov.argmax_lowest(oi.gemm(h, codes, scales))
        drafts, j = sy.plant_drafts(54, full, N, 9)
        off, n = shard_rows(N, world, rank)
        calls = []

        def partial(H, packed, M_, N_, K_, row_offset, keys_out, ws, stream):
            calls.append("partial")
            v, r = ov.shard_winners(oi.gemm(h, codes[row_offset:row_offset + N_],
                                            scales[row_offset:row_offset + N_]), row_offset)
            u = np.array([_key(v[m], r[m]) for m in range(M_)], dtype=np.uint64)
            keys_out.copy_(torch.from_numpy(u.view(np.int64)))

        def accept(keys, W, M_, draft, argmax, n_accept, bonus, stream):
            calls.append("accept")
            k = keys.view(W, M_).numpy().view(np.uint64).max(axis=0)
            a = (0xFFFFFFFF - (k & np.uint64(0xFFFFFFFF))).astype(np.int32)
            argmax.copy_(torch.from_numpy(a))
            nn, b = ov.accept(a, draft.numpy())
            n_accept.fill_(nn)
            bonus.fill_(b)

        lb.lmhead_argmax_partial, lb.lmhead_accept_keys = partial, accept
        keys_local = torch.zeros(M, dtype=torch.int64)
        keys_all = torch.zeros((world, M), dtype=torch.int64)
        argmax = torch.full((M,), -1, dtype=torch.int32)
        n_acc = torch.full((1,), -1, dtype=torch.int32)
        bonus = torch.full((1,), -1, dtype=torch.int32)
        lmhead_verify_sharded(None, None, M, n, K, off, torch.from_numpy(drafts.astype(np.int32)),
                              argmax, n_acc, bonus, None, keys_local, keys_all)
        q.put((rank, calls, argmax.tolist(), full.tolist(), int(n_acc.item()), int(bonus.item()),
               j, bool(torch.equal(keys_all[rank], keys_local))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_the_sharded_verify_sequence():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_flow, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, calls, a, full, n, b, j, own_row in got:
        assert calls == ["partial", "accept"]
        assert own_row, "the gathered keys hold each rank's own keys at its rank"
        assert a == full
        assert n == j and b == full[n]


def test_slice_key_orders_by_logit_then_lowest_row():
    vals = [-3.5, -0.0, 0.0, 1e-30, 0.25, 7.0, 7.0]
    rows = [5, 9, 8, 1, 4, 12, 3]
    keys = [_key(v, r) for v, r in zip(vals, rows)]
    best = int(np.argmax(np.array(keys, dtype=np.uint64)))
    assert (vals[best], rows[best]) == (7.0, 3)
    assert keys[0] < keys[1] < keys[2] < keys[3] < keys[4] < keys[5] < keys[6]


# ------------------------------------------------------------------------------------ GPU

torch = pytest.importorskip("torch")


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,W,j", [(16, 248_320, 4096, 2, 9), (16, 248_320, 4096, 4, 15),
                                       (16, 32_768, 4096, 3, 0), (2, 1000, 512, 2, 1),
                                       (32, 777, 256, 5, 20)])
def test_sharded_head_on_one_gpu_matches_the_oracle(M, N, K, W, j):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    from bit_weight_gemv_gb300.sharded import shard_rows
    from helpers import bf16_dev, check_argmax, dev, f16_dev
    codes, scales, h = synth.int4_problem(53, M, N, K)
    logits = oint4.gemm(h, codes, scales)
    drafts, planted = synth.plant_drafts(54, over.argmax_lowest(logits), N, j)
    H, D = bf16_dev(h), dev(drafts)
    keys = torch.zeros((W, M), dtype=torch.int64, device="cuda")
    ws = torch.zeros(lb.lmhead_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    for w in range(W):
        off, n = shard_rows(N, W, w)
        pk = torch.empty(lb.lowbit_int4_packed_bytes(n, K), dtype=torch.uint8, device="cuda")
        lb.lowbit_pack_int4(dev(np.ascontiguousarray(codes[off:off + n])),
                            f16_dev(np.ascontiguousarray(scales[off:off + n])), n, K, pk)
        lb.lmhead_argmax_partial(H, pk, M, n, K, off, keys[w], ws)
        del pk
    a = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    nacc = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    bonus = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lb.lmhead_accept_keys(keys.flip(0).contiguous(), W, M, D, a, nacc, bonus)  # any shard order
    torch.cuda.synchronize()
    got = a.cpu().numpy()
    check_argmax(got, logits, f"sharded W={W}")
    n_acc, b = int(nacc.item()), int(bonus.item())
    assert (n_acc, b) == over.accept(got, drafts)
    margins = over.top2_margin(logits)
    if np.all(margins[:planted + 1] > 1e-2):
        assert n_acc == planted
    assert not ws.any()  # the workspace is left zeroed for the next shard or call
    assert lb.lowbit_device_error() == 0
