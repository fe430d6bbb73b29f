"""Host-side expert cache of the partially resident pool (CPU only): the
eviction policies against closed forms and against Belady's optimum written
out here by brute force, and the publication rules (transactions within
capacity, misses loaded into unpublished rows, an aborted transaction leaves
the previous generation in place)."""
import numpy as np
import pytest

from w4a16_routed_expert_gb300 import build as B
from w4a16_routed_expert_gb300 import capi

POLICIES = [capi.MOE_CACHE_LRU, capi.MOE_CACHE_LFU, capi.MOE_CACHE_LRU_FREQ]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    capi.lib()


def _run_single(seq, n, C, policy, spares=0):
    """One expert demanded per forward: the cache acts as a plain cache of C."""
    c = capi.ExpertCache(n, C, spares, policy)
    hits = 0
    for e in seq:
        r = c.access([e])
        hits += r["hit"][0]
    st = c.stats()
    assert st["hits"] == hits and st["misses"] == len(seq) - hits
    return hits, st


def _belady_hits(seq, C):
    """Optimal offline replacement: on a miss with a full cache, drop the
    resident expert whose next use is farthest away (or never)."""
    cache = set()
    hits = 0
    for i, e in enumerate(seq):
        if e in cache:
            hits += 1
            continue
        if len(cache) == C:
            def next_use(x):
                for j in range(i + 1, len(seq)):
                    if seq[j] == x:
                        return j
                return len(seq) + 1
            cache.remove(max(cache, key=next_use))
        cache.add(e)
    return hits


def test_cyclic_scan_gets_no_lru_hits():
    # moe-stream, "Findings": a fixed walk over more experts than fit; LRU
    # always drops the one needed next. Every access's reuse distance is N-1
    # > C, so LRU has zero hits; Belady keeps C - 1 of them each round.
    N, C, rounds = 128, 32, 4
    seq = list(range(N)) * rounds
    hits, _ = _run_single(seq, N, C, capi.MOE_CACHE_LRU)
    assert hits == 0
    opt = _belady_hits(seq, C)
    assert opt > 0
    for p in POLICIES:
        assert _run_single(seq, N, C, p)[0] <= opt


def test_lfu_keeps_a_hot_set_that_lru_loses():
    # 12 hot experts alternate with a walk over 120 others, capacity 16. A
    # hot expert comes back after 23 other accesses of 23 distinct experts
    # (> 16): LRU misses every access. LFU counts the hot experts 10x more
    # often than the walk and keeps them once ahead: from the third round of
    # the walk on, every hot access hits.
    P, S, C = 12, 120, 16
    seq = []
    for i in range(3 * 2 * S):
        seq.append((i // 2) % P if i % 2 == 0 else P + (i // 2) % S)
    hits_lru, _ = _run_single(seq, P + S, C, capi.MOE_CACHE_LRU)
    assert hits_lru == 0
    hot_late = sum(1 for i, e in enumerate(seq) if e < P and i >= 4 * S)
    opt = _belady_hits(seq, C)
    for p in (capi.MOE_CACHE_LFU, capi.MOE_CACHE_LRU_FREQ):
        h, _ = _run_single(seq, P + S, C, p)
        assert hot_late <= h <= opt, (p, h, hot_late, opt)


def test_lru_freq_decays_every_two_capacities_of_misses():
    # F51 Nitro-MoE, "Layer 1": frequencies decay by 0.75 every 2x capacity
    # misses. A cyclic scan with N > C misses every access.
    N, C = 100, 20
    seq = list(range(N)) * 3
    hits, st = _run_single(seq, N, C, capi.MOE_CACHE_LRU_FREQ)
    assert hits == 0 and st["decays"] == len(seq) // (2 * C)
    for p in (capi.MOE_CACHE_LRU, capi.MOE_CACHE_LFU):
        assert _run_single(seq, N, C, p)[1]["decays"] == 0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_every_policy_within_the_optimum_on_skewed_traces(seed):
    rng = np.random.default_rng(seed)
    N, C = 64, 12
    w = 1.0 / np.arange(1, N + 1) ** 1.1
    seq = rng.choice(N, size=600, p=w / w.sum()).tolist()
    opt = _belady_hits(seq, C)
    for p in POLICIES:
        h, st = _run_single(seq, N, C, p)
        assert 0 <= h <= opt
        # every miss beyond the first C loads evicts one published expert
        assert st["evictions"] == max(0, st["misses"] - C)


@pytest.mark.parametrize("policy", POLICIES)
@pytest.mark.parametrize("spares", [0, 5, 16])
def test_batched_forwards_respect_capacity_and_publication(policy, spares):
    rng = np.random.default_rng(7 + policy + spares)
    N, C = 80, 16
    c = capi.ExpertCache(N, C, spares, policy)
    gen = 0
    for call in range(40):
        n = int(rng.integers(1, 3 * C))
        demanded = rng.choice(N, size=n, replace=False).tolist()
        before = {e: c.row_of(e) for e in range(N)}
        published_rows = {r for r in before.values() if r >= 0}
        res = c.access(demanded)
        # every demanded expert computed once; transactions within capacity,
        # distinct rows inside a transaction, hits only in the first one
        for t in range(res["n_txn"]):
            rows = [r for r, tt in zip(res["row"], res["txn"]) if tt == t]
            assert 0 < len(rows) <= C and len(set(rows)) == len(rows)
            assert all(0 <= r < C + spares for r in rows)
        for e, h, t, r in zip(res["experts"], res["hit"], res["txn"], res["row"]):
            assert h == (before[e] >= 0)
            if h:
                assert t == 0 and r == before[e]
        # misses of the first transaction go to rows that were not published
        # when it started, as long as enough unpublished rows exist
        misses0 = [r for e, h, t, r in zip(res["experts"], res["hit"], res["txn"], res["row"]) if t == 0 and not h]
        if len(misses0) <= C + spares - len(published_rows):
            assert not (set(misses0) & published_rows)
        # at most C experts published afterwards, each in its own row
        after = [c.row_of(e) for e in range(N)]
        pub = [r for r in after if r >= 0]
        assert len(pub) <= C and len(set(pub)) == len(pub)
        st = c.stats()
        assert st["generations"] >= gen
        gen = st["generations"]


def test_aborted_transaction_keeps_the_previous_generation():
    N, C = 40, 8
    c = capi.ExpertCache(N, C, 4, capi.MOE_CACHE_LRU)
    c.access(list(range(8)))
    gen0 = c.stats()["generations"]
    rows0 = [c.row_of(e) for e in range(N)]
    res = c.access(list(range(20, 32)), abort_txn=0)
    assert res["aborted"]
    assert [c.row_of(e) for e in range(N)] == rows0
    assert c.stats()["generations"] == gen0
    # the cache keeps working: the same request now publishes
    res = c.access(list(range(20, 32)))
    assert not res["aborted"] and c.stats()["generations"] > gen0
    assert all(c.row_of(e) >= 0 for e in range(24, 32))


def _zipf_trace(n_experts, k, tokens, s, seed):
    """Top-k routing of each token over n_experts with a Zipf(s) popularity
    (the experts of one token are distinct)."""
    rng = np.random.default_rng(seed)
    w = 1.0 / np.arange(1, n_experts + 1) ** s
    w = w / w.sum()
    return [rng.choice(n_experts, size=k, replace=False, p=w).tolist() for _ in range(tokens)]


def test_hit_rate_sweep_over_capacities(capsys):
    """Hit rate of each policy at capacities 16 / 32 / 48 / 64 / 128 on a
    synthetic top-4-of-128 trace with Zipf(1.1) popularity, one token per
    forward. LRU is a stack algorithm: its hit rate never falls when the
    capacity grows; the full capacity holds every expert after its first
    use; no policy beats the offline optimum of the flattened trace."""
    trace = _zipf_trace(128, 4, 1500, 1.1, seed=11)
    flat = [e for tok in trace for e in tok]
    rows = {}
    for p, name in zip(POLICIES, ("lru", "lfu", "lru-freq")):
        rates = []
        for C in (16, 32, 48, 64, 128):
            c = capi.ExpertCache(128, C, 0, p)
            for tok in trace:
                c.access(tok)
            st = c.stats()
            rates.append(st["hits"] / (st["hits"] + st["misses"]))
            if C == 128:
                assert st["misses"] == len(set(flat))  # only first uses miss
        rows[name] = rates
    assert all(a <= b + 1e-12 for a, b in zip(rows["lru"], rows["lru"][1:]))
    for C, i in ((16, 0), (32, 1)):
        opt = _belady_hits(flat, C) / len(flat)
        for name in rows:
            assert rows[name][i] <= opt + 1e-12, (name, C)
    with capsys.disabled():
        print("\nhit rate (top-4 of 128, Zipf 1.1, 1500 tokens) at capacity 16/32/48/64/128:")
        for name, r in rows.items():
            print(f"  {name:9s}" + " ".join(f"{v:6.3f}" for v in r))


def test_prefetched_guesses_become_hits_and_are_counted():
    # moe-stream, "Findings": the guessed experts are loaded early; a later
    # access that demands them finds them resident. Exactly the guesses that
    # are demanded before eviction count as used.
    N, C = 64, 16
    c = capi.ExpertCache(N, C, 4, capi.MOE_CACHE_LRU)
    c.access(list(range(8)))
    assert c.prefetch([20, 21, 22, 23, 3]) == 4  # 3 is resident already
    assert c.stats()["misses"] == 8  # a prefetch is not an access
    res = c.access([20, 21, 30, 3])
    hit = dict(zip(res["experts"], res["hit"]))
    assert hit == {20: 1, 21: 1, 30: 0, 3: 1}
    assert c.prefetch_stats() == dict(prefetched=4, used=2)
    c.access([20, 22])  # 20 counted once; 22 is a later use of a guess
    assert c.prefetch_stats() == dict(prefetched=4, used=3)
    with pytest.raises(ValueError):
        c.prefetch([1, 1])
