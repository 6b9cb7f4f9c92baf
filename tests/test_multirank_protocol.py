"""The multi-GPU lowering of the fused AllGather-GEMM and GEMM-ReduceScatter, played by two
`gloo` ranks on the CPU.

On one GPU the W ranks are virtual; on W GPUs each rank would own its shard and talk to its
peers through peer-mapped memory and remote signals (Triton-distributed talk: pull for the
AllGather with a ready flag per chunk and a no-overwrite barrier, push for the
ReduceScatter with a remote counter per unit; DITRON page, section 3.2: the rank-aware tile
order).  Here every rank is a process, the peers' "symmetric memory" and signals live in a
TCPStore (bytes under a key = a peer buffer, `set` = release of a flag, `add` = remote
atomic increment, `wait` with a timeout = bounded acquire poll), and numpy stands in for the
tensor cores.  What the test checks is the protocol:

* AllGather: each rank pulls the remote chunks in its transfer order (the oracle's
  ag_transfer_order), a per-chunk local flag releases each landed chunk, and the tiles run in
  the library's own tile order (dt_swizzle_plan), each waiting only for the chunks its rows
  read; the gathered bytes equal the shards bit for bit and C equals the oracle exactly
  (integer-valued inputs: every product and sum is exact in float64).
* ReduceScatter: each rank computes its partial tiles in its own scatter order (the library's
  order restricted to that source), pushes each unit's fp32 rows into the destination's slot
  for that source and increments the destination's counter; a destination reduces a unit
  when its counter reaches the oracle's expected arrivals, always in source order
  q = 0..W-1 whatever order the pushes arrived in.
* AllToAll: each rank pushes column block h of its tiles to rank h in its scatter order and
  counts every stored tile on the chunk (h, q, j) it touches; the chunk's last tile releases its
  flag (the oracle's expected counts), and rank h reads out_h once every flag is up; out_h
  equals the oracle exactly.
* A lost chunk (a flag never released) ends the consumer's bounded wait with an error on the
  host, and the ranks leave the test between steps.
"""
import datetime
import socket
import threading
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

W = 2                                   # ranks (one process each)
M, N, K = W * 150, 520, 40              # AllGather: gathered rows, columns, K
CR, BM, BN = 64, 128, 256               # chunk rows; the library's one-CTA tile
KR = 48                                 # ReduceScatter: K per rank
WAIT = datetime.timedelta(seconds=20)   # bound of every wait


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    """Integer-valued operands (exact in bf16 and in every float64 sum here)."""
    rng = np.random.Generator(np.random.PCG64(31))
    shards = [rng.integers(-3, 4, (M // W, K)).astype(np.float64) for _ in range(W)]
    b = rng.integers(-3, 4, (K, N)).astype(np.float64)
    a_rs = [rng.integers(-3, 4, (M, KR)).astype(np.float64) for _ in range(W)]
    b_rs = [rng.integers(-3, 4, (KR, N)).astype(np.float64) for _ in range(W)]
    return shards, b, a_rs, b_rs


def _lib():
    from tile_level_communication_gb300 import build
    build.build()
    import tile_level_communication_gb300 as dt
    dt.capi.lib()
    return dt


def _store(rank, port):
    return dist.TCPStore("127.0.0.1", port, W, rank == 0, timeout=WAIT)


# ------------------------------------------------------------------------------ AllGather

def _ag_rank(rank, store, dt, drop=None):
    """Rank `rank`'s fused AllGather-GEMM over the store; returns (C, pull order, tile log)."""
    from oracle import plan as oplan
    shards, b, _, _ = _inputs()
    ms = M // W
    nc = -(-ms // CR)
    epoch = b"1"
    # the producer side: this rank's shard is in its symmetric buffer from the start of the
    # call, chunk by chunk, each released by its flag
    for j in range(nc):
        lo, hi = j * CR, min((j + 1) * CR, ms)
        store.set(f"ag/mem/{rank}/{j}", shards[rank][lo:hi].tobytes())
        if (rank, j) != drop:
            store.set(f"ag/flag/{rank}/{j}", epoch)
    gather = np.full((M, K), np.nan)
    landed = {}                                   # local flags: chunk -> threading.Event
    order = oplan.ag_transfer_order(W, rank, M, CR)
    for c in order:
        landed[c] = threading.Event()
    pulled = []
    errors = []

    def puller():
        try:
            for (s, j) in order:
                lo, hi = oplan.chunk_rows_range(s, j, ms, CR)
                if s == rank:                      # local HBM: read in place, no transfer
                    gather[lo:hi] = shards[rank][lo - s * ms:hi - s * ms]
                else:
                    store.wait([f"ag/flag/{s}/{j}"], WAIT)        # acquire the peer's flag
                    assert store.get(f"ag/flag/{s}/{j}") == epoch
                    raw = store.get(f"ag/mem/{s}/{j}")           # one-sided get
                    gather[lo:hi] = np.frombuffer(raw, dtype=np.float64).reshape(hi - lo, K)
                    pulled.append((s, j))
                landed[(s, j)].set()               # release the local flag
        except Exception as e:  # noqa: BLE001 - reported to the consumer
            errors.append(e)
            for ev in landed.values():
                ev.set()

    t = threading.Thread(target=puller)
    t.start()
    args = dt.make_args(W, M, N, K, rank=rank, chunk_rows=CR, tile_m=BM)
    tile_order = dt.swizzle_plan(args, dt.OP_AG).tolist()
    tn = -(-N // BN)
    c = np.full((M, N), np.nan)
    log = []
    try:
        for tid in tile_order:
            i, n = divmod(tid, tn)
            need = oplan.tile_chunks(i, M, ms, CR, BM)     # the minimal waits of this tile
            for ch in sorted(need):
                if not landed[ch].wait(WAIT.total_seconds()) or errors:
                    raise TimeoutError(f"rank {rank}: chunk {ch} never landed "
                                       f"({errors[0] if errors else 'no flag'})")
            r0, r1 = i * BM, min((i + 1) * BM, M)
            c0, c1 = n * BN, min((n + 1) * BN, N)
            assert not np.isnan(gather[r0:r1]).any()
            c[r0:r1, c0:c1] = gather[r0:r1] @ b[:, c0:c1]
            log.append((tid, sorted(need)))
    finally:
        t.join()
    # no-overwrite barrier of pull mode: tell every peer its chunks have been read
    store.add(f"ag/read/{rank}", 1)
    return c, gather, pulled, log


def _ag_worker(rank, port, out):
    store = _store(rank, port)
    dist.init_process_group("gloo", store=store, rank=rank, world_size=W)
    dt = _lib()
    c, gather, pulled, log = _ag_rank(rank, store, dt)
    # the producer may reuse its buffer once every peer has read it
    for peer in range(W):
        if peer != rank:
            store.wait([f"ag/read/{peer}"], WAIT)
    dist.barrier()
    out[rank] = (c.tobytes(), gather.tobytes(), pulled, log)
    dist.destroy_process_group()


def test_allgather_pull_protocol_two_ranks():
    from oracle import plan as oplan
    from oracle import reference
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ag_worker, args=(port, out), nprocs=W, join=True)
        res = dict(out)
    shards, b, _, _ = _inputs()
    ref = reference.ag_gemm(shards, b)
    ms = M // W
    for rank in range(W):
        c_bytes, g_bytes, pulled, log = res[rank]
        c = np.frombuffer(c_bytes).reshape(M, N)
        assert np.array_equal(c, ref)                          # exact: integer inputs
        gathered = np.frombuffer(g_bytes).reshape(M, K)
        assert np.array_equal(gathered, reference.allgather(shards))
        want = [ch for ch in oplan.ag_transfer_order(W, rank, M, CR) if ch[0] != rank]
        assert pulled == want                                  # farthest-first pull order
        # every tile waited for exactly the chunks its rows live in, in the library's order
        tn = -(-N // BN)
        assert [t for t, _ in log] == oplan.ag_order(W, rank, M, N, CR, BM, BN)
        for tid, need in log:
            i = tid // tn
            assert set(map(tuple, need)) == oplan.tile_chunks(i, M, ms, CR, BM)


def _ag_lost_worker(rank, port, out):
    global WAIT
    store = _store(rank, port)
    dist.init_process_group("gloo", store=store, rank=rank, world_size=W)
    dt = _lib()
    WAIT = datetime.timedelta(seconds=2)
    try:
        _ag_rank(rank, store, dt, drop=(1, 1))   # rank 1 never releases its chunk 1
        out[rank] = "ok"
    except TimeoutError as e:
        out[rank] = f"timeout: {e}"
    dist.barrier()                               # both ranks leave between steps
    dist.destroy_process_group()


def test_allgather_lost_chunk_ends_the_bounded_wait():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ag_lost_worker, args=(port, out), nprocs=W, join=True)
        res = dict(out)
    assert res[0].startswith("timeout") and "(1, 1)" in res[0]   # rank 0 pulls rank 1's chunks
    assert res[1] == "ok"                                          # its own chunk is local


# ------------------------------------------------------------------------------ ReduceScatter

def _rs_units(i, ms):
    """The units m-tile i's rows split into: (s, j, row lo, row hi) per chunk piece."""
    from oracle import plan as oplan
    r0, r1 = i * BM, min((i + 1) * BM, M)
    out = []
    g = r0
    while g < r1:
        s, j = oplan.chunk_of_row(g, ms, CR)
        hi = min(r1, oplan.chunk_rows_range(s, j, ms, CR)[1])
        out.append((s, j, g, hi))
        g = hi
    return out


def _rs_worker(rank, port, out):
    from oracle import plan as oplan
    store = _store(rank, port)
    dist.init_process_group("gloo", store=store, rank=rank, world_size=W)
    dt = _lib()
    _, _, a_rs, b_rs = _inputs()
    ms = M // W
    tm, tn = -(-M // BM), -(-N // BN)
    args = dt.make_args(W, M, N, KR, chunk_rows=CR, tile_m=BM)
    full = dt.swizzle_plan(args, dt.OP_RS).tolist()
    mine = [t for t in full if t // (tm * tn) == rank]       # this source's scatter order
    expected = oplan.rs_expected_arrivals(W, M, N, CR, BM, BN)
    my_units = [u for u in expected if u[1] == rank]          # units this rank reduces
    result = np.full((ms, N), np.nan, dtype=np.float32)
    errors = []

    def reducer():
        try:
            pending = set(my_units)
            while pending:
                done = []
                for (i, s, j, n) in sorted(pending):
                    key = f"rs/cnt/{s}/{i}/{j}/{n}"
                    if not store.check([key]) or store.add(key, 0) < expected[(i, s, j, n)]:
                        continue
                    # every partial is in: fold them in the fixed source order q = 0..W-1
                    lo = max(i * BM, oplan.chunk_rows_range(s, j, ms, CR)[0])
                    hi = min((i + 1) * BM, M, oplan.chunk_rows_range(s, j, ms, CR)[1])
                    c0, c1 = n * BN, min((n + 1) * BN, N)
                    acc = None
                    for q in range(W):
                        raw = store.get(f"rs/recv/{s}/{q}/{i}/{j}/{n}")
                        part = np.frombuffer(raw, dtype=np.float32).reshape(hi - lo, c1 - c0)
                        acc = part.copy() if acc is None else (acc + part).astype(np.float32)
                    result[lo - s * ms:hi - s * ms, c0:c1] = acc
                    done.append((i, s, j, n))
                pending -= set(done)
                if not done:
                    time.sleep(0.001)
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    t = threading.Thread(target=reducer)
    t.start()
    sent = []                                  # per tile: the units it pushed
    for tid in mine:
        q, rem = divmod(tid, tm * tn)
        i, n = divmod(rem, tn)
        r0, r1 = i * BM, min((i + 1) * BM, M)
        c0, c1 = n * BN, min((n + 1) * BN, N)
        p = (a_rs[q][r0:r1] @ b_rs[q][:, c0:c1]).astype(np.float32)   # fp32 partial tile
        units = []
        for (s, j, lo, hi) in _rs_units(i, ms):
            # push: the unit's rows into destination s's slot for source q, then the counter
            store.set(f"rs/recv/{s}/{q}/{i}/{j}/{n}", p[lo - r0:hi - r0].tobytes())
            store.add(f"rs/cnt/{s}/{i}/{j}/{n}", 1)
            units.append((s, j))
        sent.append(units)
    t.join(timeout=WAIT.total_seconds())
    assert not t.is_alive() and not errors, errors
    dist.barrier()
    out[rank] = (result.tobytes(), sent, mine)
    dist.destroy_process_group()


def test_reducescatter_push_protocol_two_ranks():
    from oracle import plan as oplan
    from oracle import reference
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rs_worker, args=(port, out), nprocs=W, join=True)
        res = dict(out)
    _, _, a_rs, b_rs = _inputs()
    ref = reference.gemm_rs(a_rs, b_rs)
    ms = M // W
    # the fp32 partials and their source-order sum, computed directly
    parts = [(a_rs[q] @ b_rs[q]).astype(np.float32) for q in range(W)]
    fold = parts[0].copy()
    for q in range(1, W):
        fold = (fold + parts[q]).astype(np.float32)
    tm, tn = -(-M // BM), -(-N // BN)
    for s in range(W):
        got_bytes, sent, mine = res[s]
        got = np.frombuffer(got_bytes, dtype=np.float32).reshape(ms, N)
        assert np.array_equal(got, fold[s * ms:(s + 1) * ms])   # fixed-order fp32 fold, bitwise
        assert np.array_equal(got.astype(np.float64), ref[s])  # exact: integer inputs
        # each source sent in its own scatter order: the library's order restricted to it
        assert mine == [t for t in oplan.rs_order(W, M, N, CR, BM, BN) if t // (tm * tn) == s]
        # a source's first tile feeds the first chunk of the rank after it (send order q+1 first,
        # its own block last), and its last tile feeds its own block
        assert ((s + 1) % W, 0) in sent[0]
        assert s in {d for d, _ in sent[-1]}
        assert all(any(d == (s + 1) % W for d, _ in units) for units in sent[:1])


# ------------------------------------------------------------------------------ AllToAll

A2A_MS, A2A_NW, A2A_K, A2A_CR = 150, 264, 40, 64   # rows per rank, columns per destination


def _a2a_inputs():
    rng = np.random.Generator(np.random.PCG64(33))
    a = [rng.integers(-3, 4, (A2A_MS, A2A_K)).astype(np.float64) for _ in range(W)]
    b = [rng.integers(-3, 4, (A2A_K, W * A2A_NW)).astype(np.float64) for _ in range(W)]
    return a, b


def _a2a_worker(rank, port, out):
    """Rank `rank` pushes column block h of its own tiles to rank h, in its scatter order, and
    counts each stored tile on the chunk (h, q, j) its rows touch; the chunk's last tile
    releases the chunk's flag on rank h.  Rank h waits for every chunk's flag, then reads its
    out_h."""
    from oracle import plan as oplan
    store = _store(rank, port)
    dist.init_process_group("gloo", store=store, rank=rank, world_size=W)
    dt = _lib()
    a, b = _a2a_inputs()
    n = W * A2A_NW
    args = dt.make_args(W, W * A2A_MS, n, A2A_K, chunk_rows=A2A_CR, tile_m=BM)
    full = dt.swizzle_plan(args, dt.OP_A2A).tolist()
    nw, nc, tm, tnw = oplan.a2a_geometry(W, A2A_MS, n, A2A_CR, BM, BN)
    tn = W * tnw
    mine = [t for t in full if t // (tm * tn) == rank]
    expected = oplan.a2a_expected_counts(W, A2A_MS, n, A2A_CR, BM, BN)
    sent = []
    for tid in mine:
        q, rem = divmod(tid, tm * tn)
        i, c_all = divmod(rem, tn)
        h, c = divmod(c_all, tnw)
        r0, r1 = i * BM, min((i + 1) * BM, A2A_MS)
        c0, c1 = h * nw + c * BN, min(h * nw + (c + 1) * BN, (h + 1) * nw)
        y = a[q][r0:r1] @ b[q][:, c0:c1]
        # push: the tile's rows into out_h, rows q * Ms + r, columns c0 - h * Nw ..
        store.set(f"a2a/out/{h}/{q}/{i}/{c}", y.tobytes())
        for j in range(r0 // A2A_CR, (r1 - 1) // A2A_CR + 1):
            done = store.add(f"a2a/cnt/{h}/{q}/{j}", 1)
            if done == expected[(h, q, j)]:
                store.set(f"a2a/flag/{h}/{q}/{j}", b"1")   # release: chunk (h, q, j) complete
        sent.append(h)
    # the consumer side: rank h's out_h, once every source's chunks are flagged
    res = np.full((W * A2A_MS, nw), np.nan)
    for q in range(W):
        for j in range(nc):
            store.wait([f"a2a/flag/{rank}/{q}/{j}"], WAIT)
        for i in range(tm):
            for c in range(tnw):
                r0, r1 = i * BM, min((i + 1) * BM, A2A_MS)
                c0, c1 = c * BN, min((c + 1) * BN, nw)
                raw = store.get(f"a2a/out/{rank}/{q}/{i}/{c}")
                res[q * A2A_MS + r0:q * A2A_MS + r1, c0:c1] = \
                    np.frombuffer(raw).reshape(r1 - r0, c1 - c0)
    dist.barrier()
    out[rank] = (res.tobytes(), sent)
    dist.destroy_process_group()


def test_alltoall_push_protocol_two_ranks():
    from oracle import plan as oplan
    from oracle import reference
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_a2a_worker, args=(port, out), nprocs=W, join=True)
        res = dict(out)
    a, b = _a2a_inputs()
    ref = reference.gemm_a2a(a, b)
    for h in range(W):
        got_bytes, sent = res[h]
        got = np.frombuffer(got_bytes).reshape(W * A2A_MS, A2A_NW)
        assert np.array_equal(got, ref[h])                       # exact: integer inputs
        # rank h sends to h+1 first and keeps its own block for last
        assert sent[0] == (h + 1) % W and sent[-1] == h
        assert sent == sorted(sent, key=lambda d: oplan.rs_dpos(h, d, W))
