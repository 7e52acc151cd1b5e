"""The native page allocator / continuous-batching scheduler (no GPU).

* matches the reference model of the admission policy (``oracle/admission.py``) step by
  step, bit for bit: admissions, retirements, appended tokens, slot mappings in every
  layer, decode batches, context lengths and block tables - on the 1000-step trace, on a
  small pool that makes requests wait, and with several layers;
* invariants: pages never shared, never more pages than credits, the free list returns
  to full, contexts never exceed the limit;
* rejection of a request larger than the pool, clamping of the new-token budget, and
  the --stats counters on a hand-checked example.
"""
import numpy as np
import pytest

from oracle.admission import AdmissionModel, Rejected
from workloads import configs


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_180_gb300 import build
    build.build()
    import paged_kv_cache_180_gb300 as p
    return p


def _run_both(pkv, num_pages, num_layers, num_slots, requests, steps, free_order=None, max_context=2048):
    native = pkv.Scheduler(num_pages, num_layers, 16, max_context, num_slots, free_order)
    model = AdmissionModel(num_pages, num_layers, 16, max_context, num_slots, free_order)
    for rid, (p, n) in enumerate(requests):
        native.submit(rid, p, n)
        model.submit(rid, p, n)
    plans = []
    for step in range(steps):
        a = native.step()
        b = model.step()
        for key in ("finished", "admitted", "admitted_slot", "append_request", "append_position", "decode_slot",
                    "context_lens"):
            assert list(a[key]) == list(b[key]), (step, key)
        assert np.array_equal(a["append_slot_mapping"], np.array(b["append_slot_mapping"], dtype=np.int32).reshape(
            num_layers, -1)), step
        assert np.array_equal(a["block_tables"], np.array(b["block_tables"], dtype=np.int32)), step
        plans.append(a)
    return native, model, plans


def _check_invariants(plans, num_pages, num_layers, max_context=2048):
    for pl in plans:
        used = pl["block_tables"][pl["block_tables"] >= 0]
        assert len(np.unique(used)) == used.size          # a page belongs to one (slot, layer, block)
        assert used.size <= num_pages
        assert (pl["context_lens"] <= max_context).all()


def test_trace_matches_reference_model(pkv):
    tr = configs.trace()
    reqs = list(zip(tr.prompt_lens.tolist(), tr.new_budgets.tolist()))
    native, model, plans = _run_both(pkv, tr.num_pages, 1, tr.num_slots, reqs, tr.num_steps, tr.free_order)
    _check_invariants(plans, tr.num_pages, 1)
    st = native.stats()
    assert st["peak_active"] == model.stats["peak_active"] == 32       # slot-bound with a 4096-page pool
    assert st["largest_batch"] == model.stats["largest_batch"]
    assert st["peak_pages"] == model.stats["peak_pages"]
    assert st["admission_waits"] == model.stats["admission_waits"] == 0
    assert sum(len(p["finished"]) for p in plans) > 50


def test_small_pool_waits_match(pkv):
    tr = configs.trace(num_pages=512)
    reqs = list(zip(tr.prompt_lens.tolist(), tr.new_budgets.tolist()))
    order = configs.trace(num_pages=512).free_order
    native, model, plans = _run_both(pkv, 512, 1, 32, reqs, 600, order)
    _check_invariants(plans, 512, 1)
    st = native.stats()
    assert st["admission_waits"] == model.stats["admission_waits"] > 0
    assert st["peak_pages"] <= 512 and st["credits_in_use"] <= 512


def test_multi_layer_matches(pkv):
    r = np.random.default_rng(7)
    reqs = [(int(r.integers(1, 200)), int(r.integers(1, 60))) for _ in range(40)]
    native, model, plans = _run_both(pkv, 600, 4, 6, reqs, 200, np.random.default_rng(8).permutation(600))
    _check_invariants(plans, 600, 4)


def test_all_pages_come_back(pkv):
    reqs = [(17, 3), (1, 1), (64, 10), (5, 40)]
    native, model, plans = _run_both(pkv, 40, 2, 2, reqs, 80)
    st = native.stats()
    assert st["free_pages"] == 40 and st["active"] == 0 and st["queued"] == 0 and st["credits_in_use"] == 0


def test_rejection_and_clamp(pkv):
    s = pkv.Scheduler(100, 1, 16, 2048, 4)
    with pytest.raises(pkv.PkvError) as e:
        s.submit(0, 1601, 10)                 # ceil(1610 / 16) = 101 pages > 100
    assert e.value.code == -9
    m = AdmissionModel(100)
    with pytest.raises(Rejected):
        m.submit(0, 1601, 10)
    with pytest.raises(pkv.PkvError):
        s.submit(1, 1500, 10000)              # budget clamped to 2048 - 1500 + 1 = 549 -> 128 pages > 100
    big = pkv.Scheduler(200, 1, 16, 2048, 4)
    big.submit(1, 1500, 10000)
    plan = big.step()
    assert plan["context_lens"][0] == 1501     # prompt + its first decode token
    for _ in range(600):
        plan = big.step()
    assert big.stats()["active"] == 0          # decoded 548 tokens: context ended at 2048
    for bad in ((0, 5), (2049, 1), (10, 0)):
        with pytest.raises(pkv.PkvError):
            s.submit(9, *bad)


def test_stats_hand_example(pkv):
    # Pool of 8 pages, 4 slots.  Step 0 admits r0 (20+5-1 -> 2 credits) and r1 (33+1-1 -> 3);
    # r2 (60+8-1 -> 5) waits; step 1 retires r1 (budget 1), admits r2 into slot 1 and r3 into slot 2.
    s = pkv.Scheduler(8, 1, 16, 2048, 4)
    for rid, (p, n) in enumerate([(20, 5), (33, 1), (60, 8), (5, 2)]):
        s.submit(rid, p, n)
    p0 = s.step()
    assert list(p0["admitted"]) == [0, 1] and list(p0["decode_slot"]) == [0]
    p1 = s.step()
    assert list(p1["finished"]) == [1] and list(p1["admitted"]) == [2, 3] and list(p1["admitted_slot"]) == [1, 2]
    # LIFO: r1's pages (free list order 5, 4, 3 pushed in block order) go to r2 as 3, 4, 5, then 2
    assert list(p1["block_tables"][1, 0, :4]) == [3, 4, 5, 2]
    for _ in range(10):
        s.step()
    st = s.stats()
    assert st == dict(pool_pages=8, peak_active=3, largest_batch=3, peak_pages=7, admission_waits=1, free_pages=8,
                      credits_in_use=0, active=0, queued=0, steps=12)


@pytest.mark.parametrize("seed", range(24))
def test_random_configurations_match_and_drain(pkv, seed):
    """Seeded random pools, layer counts, slot counts, context limits and request mixes (some
    requests too large for the pool, some budgets clamped): the native scheduler matches the
    reference model at every step, the invariants hold, and every page comes back."""
    r = np.random.default_rng(9000 + seed)
    num_pages = int(r.integers(8, 160))
    num_layers = int(r.integers(1, 4))
    num_slots = int(r.integers(1, 9))
    max_context = int(r.choice([64, 256, 2048]))
    free_order = [int(x) for x in r.permutation(num_pages)] if seed % 2 else None
    native = pkv.Scheduler(num_pages, num_layers, 16, max_context, num_slots, free_order)
    model = AdmissionModel(num_pages, num_layers, 16, max_context, num_slots, free_order)
    accepted = []
    for rid in range(int(r.integers(3, 16))):
        p = int(r.integers(1, max_context + 1))
        n = int(r.integers(1, 80))
        try:
            model.submit(rid, p, n)
        except Rejected:
            with pytest.raises(pkv.PkvError):
                native.submit(rid, p, n)
            continue
        native.submit(rid, p, n)
        accepted.append((p, n))
    work = sum(min(n, max_context - p + 1) for p, n in accepted)
    plans = []
    for step in range(work + len(accepted) + 8):
        a = native.step()
        b = model.step()
        for key in ("finished", "admitted", "admitted_slot", "append_request", "append_position", "decode_slot",
                    "context_lens"):
            assert list(a[key]) == list(b[key]), (seed, step, key)
        assert np.array_equal(a["block_tables"], np.array(b["block_tables"], dtype=np.int32)), (seed, step)
        plans.append(a)
    _check_invariants(plans, num_pages, num_layers, max_context)
    st = native.stats()
    assert st["free_pages"] == num_pages and st["active"] == 0 and st["queued"] == 0 and st["credits_in_use"] == 0
