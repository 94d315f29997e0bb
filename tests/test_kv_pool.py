"""Host tests of the paged-KV block allocator (include/mk_kv.h): page accounting under
random admit / grow / evict sequences, the FIFO free-list order, and argument checks.
No GPU."""
import numpy as np
import pytest

import workloads as W
import persistent_moe_decode_megakernel_gb300 as mk


@pytest.fixture(scope="module", autouse=True)
def built():
    mk.build()


def _check_invariants(pool, num_pages, max_slots, ps):
    live = [s for s in range(max_slots) if pool.length(s) >= 0]
    lens, bt = pool.fill(live) if live else (np.zeros(0, np.int32), np.zeros((0, pool.max_pages), np.int32))
    used = []
    for i, s in enumerate(live):
        n = -(-int(lens[i]) // ps)
        assert np.all(bt[i, :n] >= 0) and np.all(bt[i, n:] == -1)   # exactly the pages covering the length
        used.extend(bt[i, :n].tolist())
    assert len(used) == len(set(used))                               # no page held twice
    assert len(used) + pool.free_pages() == num_pages                # nothing lost


def test_admission_in_order_reproduces_the_dealt_block_tables():
    lens = [65, 1, 300, 17, 16, 512, 2, 90]
    ps, num_pages, mpp = 16, 200, 40
    bt_ref, free_ref = W.make_block_tables(lens, ps, num_pages, mpp)
    perm = np.concatenate([bt_ref.numpy()[b, :-(-L // ps)] for b, L in enumerate(lens)] + [np.array(free_ref)])
    pool = mk.KvPool(num_pages, ps, 8, mpp, order=perm)
    slots = [pool.admit(L) for L in lens]
    assert slots == list(range(8))
    got_lens, got_bt = pool.fill(slots)
    assert np.array_equal(got_lens, lens) and np.array_equal(got_bt, bt_ref.numpy())
    assert pool.free_pages() == len(free_ref)


def test_fifo_free_list_growth_and_eviction():
    pool = mk.KvPool(10, 4, 3, 10)
    a = pool.admit(5)                      # pages 0, 1
    b = pool.admit(4)                      # page 2
    pool.reserve(b, 5)                     # crosses into page 3
    pool.evict(a)                          # 0, 1 go to the tail: free = 4..9, 0, 1
    c = pool.admit(24)                     # six pages from the head: 4..9
    assert c == a == 0
    _, bt = pool.fill([c, b])
    assert bt[0, :6].tolist() == [4, 5, 6, 7, 8, 9] and bt[1, :2].tolist() == [2, 3]
    pool.reserve(c, 25)                    # the next free page is 0
    assert pool.fill([c])[1][0, 6] == 0
    assert pool.free_pages() == 1


@pytest.mark.parametrize("seed", range(5))
def test_random_workload_keeps_every_page_accounted(seed):
    rng = np.random.default_rng(seed)
    num_pages, ps, max_slots, mpp = 64, 8, 6, 12
    pool = mk.KvPool(num_pages, ps, max_slots, mpp, order=rng.permutation(num_pages))
    for _ in range(400):
        op = rng.integers(3)
        live = [s for s in range(max_slots) if pool.length(s) >= 0]
        before = (pool.free_pages(), [pool.length(s) for s in range(max_slots)])
        try:
            if op == 0:
                pool.admit(int(rng.integers(1, ps * mpp + 1)))
            elif op == 1 and live:
                s = int(rng.choice(live))
                pool.reserve(s, pool.length(s) + int(rng.integers(0, 3 * ps)))
            elif op == 2 and live:
                pool.evict(int(rng.choice(live)))
        except mk.MkError as e:
            # a failing call changes nothing
            assert e.code in (mk.MK_ERR_OOM, mk.MK_ERR_INVALID_ARG)
            assert (pool.free_pages(), [pool.length(s) for s in range(max_slots)]) == before
        _check_invariants(pool, num_pages, max_slots, ps)


def test_argument_checks():
    with pytest.raises(mk.MkError):
        mk.KvPool(0, 16, 4, 4)
    with pytest.raises(mk.MkError):
        mk.KvPool(4, 16, 4, 4, order=[0, 1, 1, 3])      # not a permutation
    pool = mk.KvPool(4, 16, 2, 2)
    with pytest.raises(mk.MkError):
        pool.admit(0)
    with pytest.raises(mk.MkError):
        pool.admit(33)                                   # more pages than a slot may hold
    s = pool.admit(16)
    with pytest.raises(mk.MkError):
        pool.reserve(s, 15)                              # shrinking
    with pytest.raises(mk.MkError):
        pool.fill([s, s])                                # listed twice
    with pytest.raises(mk.MkError):
        pool.evict(1)                                    # not live
    pool.admit(32)
    with pytest.raises(mk.MkError) as e:
        pool.admit(1)                                    # no slot left
    assert e.value.code == mk.MK_ERR_OOM
