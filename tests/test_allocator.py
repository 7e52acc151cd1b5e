"""The native page allocator (``pkv_alloc_*``) on its own (no GPU).

* Replays the reference model of the admission policy (``oracle/admission.py``) through the
  allocator calls - admit for each admission, one page lookup per appended token and layer,
  free_seq for each retirement - and checks the slot of every appended token, the block
  tables, the free-list size and the credits after every step; when the model makes the
  queue head wait, the allocator refuses the same request with PKV_ERR_NO_CREDIT.
* A hand-checked example of the LIFO free list, and every error code.
"""
import numpy as np
import pytest

from oracle.admission import AdmissionModel
from workloads import configs


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_180_gb300 import build
    build.build()
    import paged_kv_cache_180_gb300 as p
    return p


def _replay(pkv, num_pages, num_layers, num_slots, requests, steps, free_order=None, max_context=2048):
    model = AdmissionModel(num_pages, num_layers, 16, max_context, num_slots, free_order)
    alloc = pkv.Allocator(num_pages, num_layers, 16, max_context, num_slots, free_order)
    info = {}
    for rid, (p, n) in enumerate(requests):
        model.submit(rid, p, n)
        info[rid] = (p, n)
    slot_of = {}
    waits_seen = 0
    for step in range(steps):
        waits_before = model.stats["admission_waits"]
        plan = model.step()
        for rid in plan["finished"]:
            alloc.free_seq(slot_of.pop(rid))
        for rid, slot in zip(plan["admitted"], plan["admitted_slot"]):
            rc, credits = alloc.admit(slot, *info[rid])
            assert rc == alloc.OK, (step, rid)
            assert credits == model.slot[slot]["credits"]
            slot_of[rid] = slot
        for i, (rid, pos) in enumerate(zip(plan["append_request"], plan["append_position"])):
            for layer in range(num_layers):
                page = alloc.page(slot_of[rid], layer, pos // 16)
                assert page * 16 + pos % 16 == plan["append_slot_mapping"][layer][i], (step, i, layer)
        assert np.array_equal(alloc.block_tables(), np.array(plan["block_tables"], dtype=np.int32)), step
        free, credits_used = alloc.state()
        assert free == len(model.free) and credits_used == model.credits_used, step
        if model.stats["admission_waits"] > waits_before:
            # the queue head waited for credits with a slot free: the allocator refuses it too
            head = model.queue[0]
            free_slot = next(s for s in range(num_slots) if model.slot[s] is None)
            rc, credits = alloc.admit(free_slot, head["prompt"], head["new"])
            assert rc == alloc.NO_CREDIT and credits == head["credits"]
            assert alloc.state() == (free, credits_used)          # nothing was reserved
            waits_seen += 1
    return waits_seen


def test_trace_replayed_through_the_allocator(pkv):
    tr = configs.trace()
    reqs = list(zip(tr.prompt_lens.tolist(), tr.new_budgets.tolist()))
    _replay(pkv, tr.num_pages, 1, tr.num_slots, reqs, tr.num_steps, tr.free_order)


def test_small_pool_waits_replayed_through_the_allocator(pkv):
    tr = configs.trace(num_pages=512)
    reqs = list(zip(tr.prompt_lens.tolist(), tr.new_budgets.tolist()))
    assert _replay(pkv, 512, 1, 32, reqs, 600, tr.free_order) > 0


@pytest.mark.parametrize("seed", range(6))
def test_random_configurations_replayed_through_the_allocator(pkv, seed):
    r = np.random.default_rng(1000 + seed)
    layers = int(r.integers(1, 5))
    slots = int(r.integers(1, 12))
    max_context = int(r.choice([64, 300, 2048]))
    pages = int(r.integers(max_context // 16 * layers, 6 * max_context // 16 * layers + 1))
    n_req = int(r.integers(5, 60))
    prompts = r.integers(1, max_context + 1, n_req)
    news = r.integers(1, max_context + 1, n_req)
    order = r.permutation(pages).astype(np.int32)
    _replay(pkv, pages, layers, slots, list(zip(prompts.tolist(), news.tolist())), 400, order, max_context)


def test_hand_checked_lifo_example(pkv):
    a = pkv.Allocator(4, 1, 16, 64, 2, free_order=[3, 1, 0, 2])
    rc, credits = a.admit(0, 20, 5)            # prefix 24 tokens -> 2 pages in 1 layer
    assert (rc, credits) == (a.OK, 2)
    assert a.page(0, 0, 0) == 2                 # popped from the back
    assert a.page(0, 0, 1) == 0
    assert a.page(0, 0, 0) == 2                 # assigned already: no pop
    assert a.state() == (2, 2)
    a.free_seq(0)                               # pushes 2 then 0
    assert a.state() == (4, 0)
    rc, _ = a.admit(1, 1, 1)
    assert rc == a.OK and a.page(1, 0, 0) == 0 and a.page(1, 0, 1) == 2 and a.page(1, 0, 2) == 1
    assert (a.block_tables()[1, 0, :4] == [0, 2, 1, -1]).all() and (a.block_tables()[0] == -1).all()


def test_credits_clamp_reject_and_wait(pkv):
    a = pkv.Allocator(8, 2, 16, 64, 3)
    # prompt 60 + new 100 clamps to new = 5: prefix 64 -> 4 pages x 2 layers = 8 credits (the whole pool)
    assert a.admit(0, 60, 100) == (a.OK, 8)
    assert a.admit(1, 1, 1) == (a.NO_CREDIT, 2)     # fits the pool, not beside seq 0: wait
    assert a.state() == (8, 8)
    a.free_seq(0)
    assert a.admit(1, 1, 1) == (a.OK, 2)
    b = pkv.Allocator(7, 2, 16, 64, 1)
    assert b.admit(0, 60, 100) == (b.EXCEEDS_POOL, 8)   # more credits than the whole pool
    assert b.state() == (7, 0)


def test_error_codes(pkv):
    a = pkv.Allocator(2, 1, 16, 64, 2)
    with pytest.raises(pkv.PkvError) as e:
        a.page(0, 0, 0)                         # not admitted
    assert e.value.code == -11
    with pytest.raises(pkv.PkvError) as e:
        a.free_seq(1)
    assert e.value.code == -11
    assert a.admit(0, 1, 1)[0] == a.OK
    with pytest.raises(pkv.PkvError) as e:
        a.admit(0, 1, 1)                        # admitted already
    assert e.value.code == -11
    for args in ((2, 1, 1), (-1, 1, 1), (1, 0, 1), (1, 65, 1), (1, 1, 0)):
        with pytest.raises(pkv.PkvError) as e:
            a.admit(*args)
        assert e.value.code == -2
    for args in ((0, 1, 0), (0, 0, 4), (0, 0, -1), (3, 0, 0)):
        with pytest.raises(pkv.PkvError) as e:
            a.page(*args)
        assert e.value.code == -2
    # pages beyond the credits come from the free list until it runs dry
    assert a.page(0, 0, 0) >= 0 and a.page(0, 0, 1) >= 0
    with pytest.raises(pkv.PkvError) as e:
        a.page(0, 0, 2)
    assert e.value.code == -10                  # PKV_ERR_NO_PAGE
    for bad in ([0, 0], [0, 2], [-1, 0]):
        with pytest.raises(pkv.PkvError) as e:
            pkv.Allocator(2, 1, 16, 64, 1, free_order=bad)
        assert e.value.code == -2
    assert pkv.status_string(-13).startswith("request credits")
