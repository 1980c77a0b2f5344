"""GPU vs oracle for the chained whole-model apply (a receiver several
versions behind applies the patches it missed in one pass): chains of real
encode patches and of random patches with overlapping index sets, dense and
sparse chunks, ragged and empty tensors, unaligned receivers, chains longer
than one launch takes, and the error contract. Every comparison is
bit-exact against the oracle applying the patches one after the other."""
import numpy as np
import pytest
import torch

import oracle
import rl_post_trainer_gb300 as pulse
from pulse_testutil import Guarded, dev_u16, dev_u32, host_u16

pytestmark = pytest.mark.gpu

CHUNK = 8192  # elements per chunk of the chunk-owned apply
SIZES = [0, 1, 7, CHUNK - 1, CHUNK, CHUNK + 1, 3 * CHUNK + 100, 200003]


def _dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return torch.device("cuda", 0)


def _encode_chain(rng, n, etas):
    """w0 and the patches of successive versions of one tensor: an FP32
    master moved by eta * z per version, each version encoded against the
    last by the oracle."""
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    prev = oracle.bf16_rne(master.view(np.uint32)).astype(np.uint16) if n else np.zeros(0, np.uint16)
    w0 = prev.copy()
    patches = []
    for eta in etas:
        master = (master + np.float32(eta) * rng.standard_normal(n).astype(np.float32)).astype(np.float32)
        idx, val = oracle.encode(master, prev)
        patches.append((idx, val))
    return w0, patches, prev


def _rand_patch(rng, n, k):
    k = min(k, n)
    idx = np.sort(rng.choice(n, size=k, replace=False)).astype(np.uint32) if k else np.zeros(0, np.uint32)
    return idx, rng.integers(0, 1 << 16, size=k).astype(np.uint16)


def _dev_patch(p, dev):
    idx, val = p
    if idx.size == 0:
        return (torch.empty(0, dtype=torch.int32, device=dev),
                torch.empty(0, dtype=torch.int16, device=dev), 0)
    return dev_u32(idx, dev), dev_u16(val, dev), idx.size


def _run(w0s, chains, dev, offset=0):
    """chains[t] = list of patches of tensor t (oldest first). Returns the
    GPU result per tensor and the plan's error word."""
    ws, guards = [], []
    for w0 in w0s:
        g = Guarded(w0.size + offset, torch.int16, dev)
        guards.append(g)
        v = g.t[offset:]
        if w0.size:
            v.copy_(dev_u16(w0, dev))
        ws.append(v)
    slots = [pulse.TensorSlot(w0.size, w=w) for w0, w in zip(w0s, ws)]
    nv = len(chains[0])
    patches = [[_dev_patch(chains[t][v], dev) for t in range(len(w0s))] for v in range(nv)]
    with pulse.Plan(slots) as plan:
        plan.apply_chain(patches)
        torch.cuda.synchronize()
        err = plan.get_error()
    for g in guards:
        g.check("w")
    return [host_u16(w) for w in ws], err


def _expect(w0s, chains):
    out = []
    for w0, chain in zip(w0s, chains):
        w = w0.copy()
        for idx, val in chain:
            oracle.apply(w, idx, val)
        out.append(w)
    return out


@pytest.mark.parametrize("nv", [1, 2, 4, 5])
def test_encode_chain_matches_oracle(nv):
    dev = _dev()
    rng = np.random.default_rng(100 + nv)
    etas = [3e-6, 1e-7, 1e-4, 3e-6, 3e-7][:nv]  # ~8 %, ~0.5 %, ~70 %, ... changed per version
    w0s, chains, finals = [], [], []
    for n in SIZES:
        w0, patches, last = _encode_chain(rng, n, etas)
        w0s.append(w0)
        chains.append(patches)
        finals.append(last)
    got, err = _run(w0s, chains, dev)
    assert err == 0
    for g, e, f in zip(got, _expect(w0s, chains), finals):
        np.testing.assert_array_equal(g, e)
        np.testing.assert_array_equal(g, f)  # the receiver ends at the trainer's last view


def test_random_chain_overlapping_and_composed():
    """Random patches whose index sets overlap across versions: the later
    value must win; the result also equals the oracle's composed patch."""
    dev = _dev()
    rng = np.random.default_rng(7)
    sizes = [5 * CHUNK + 33, 70000, 9]
    w0s = [rng.integers(0, 1 << 16, size=n).astype(np.uint16) for n in sizes]
    ks = [(4000, 20000, 60000), (30, 2, 0), (9, 9, 1)]
    chains = []
    for n, kk in zip(sizes, ks):
        chains.append([_rand_patch(rng, n, k) for k in kk])
    got, err = _run(w0s, chains, dev)
    assert err == 0
    for g, e, w0, chain in zip(got, _expect(w0s, chains), w0s, chains):
        np.testing.assert_array_equal(g, e)
        ci, cv = oracle.compose_chain(chain)
        w = w0.copy()
        oracle.apply(w, ci, cv)
        np.testing.assert_array_equal(g, w)


def test_identical_index_sets_last_wins():
    dev = _dev()
    rng = np.random.default_rng(11)
    n = 4 * CHUNK
    idx = np.sort(rng.choice(n, size=20000, replace=False)).astype(np.uint32)
    chain = [(idx, np.full(idx.size, v, np.uint16)) for v in (1, 2, 3)]
    w0 = np.zeros(n, np.uint16)
    (got,), err = _run([w0], [chain], dev)
    assert err == 0
    exp = np.zeros(n, np.uint16)
    exp[idx] = 3
    np.testing.assert_array_equal(got, exp)


def test_longer_than_one_launch():
    """Seventeen versions: the library takes them in two launches."""
    dev = _dev()
    rng = np.random.default_rng(17)
    sizes = [3 * CHUNK + 5, 1000]
    w0s, chains = [], []
    for n in sizes:
        w0, patches, _ = _encode_chain(rng, n, [3e-6] * 17)
        w0s.append(w0)
        chains.append(patches)
    got, err = _run(w0s, chains, dev)
    assert err == 0
    for g, e in zip(got, _expect(w0s, chains)):
        np.testing.assert_array_equal(g, e)


@pytest.mark.parametrize("offset", [1, 3])
def test_unaligned_receiver(offset):
    """w not 16-byte aligned: every chunk takes the direct-store path."""
    dev = _dev()
    rng = np.random.default_rng(30 + offset)
    w0s, chains = [], []
    for n in (2 * CHUNK + 17, 333):
        w0, patches, _ = _encode_chain(rng, n, [1e-5, 3e-6, 1e-4])
        w0s.append(w0)
        chains.append(patches)
    got, err = _run(w0s, chains, dev, offset=offset)
    assert err == 0
    for g, e in zip(got, _expect(w0s, chains)):
        np.testing.assert_array_equal(g, e)


def test_errors_reported():
    dev = _dev()
    n = 3 * CHUNK
    w0 = np.zeros(n, np.uint16)
    gi = np.arange(0, n, 5, dtype=np.uint32)
    good = (gi, np.ones(gi.size, np.uint16))
    # an entry out of order: it lies outside the chunk the partition gives it
    bad_idx = good[0].copy()
    bad_idx[10] = n - 1
    _, err = _run([w0], [[good, (bad_idx, good[1])]], dev)
    assert err == pulse.pulse.PULSE_ERR_INDEX
    # a count above n is clamped and reported
    ws = torch.zeros(10, dtype=torch.int16, device=dev)
    idx = torch.arange(12, dtype=torch.int32, device=dev)
    val = torch.ones(12, dtype=torch.int16, device=dev)
    with pulse.Plan([pulse.TensorSlot(10, w=ws)]) as plan:
        plan.apply_chain([[(idx, val, 12)]])
        torch.cuda.synchronize()
        assert plan.get_error() == pulse.pulse.PULSE_ERR_INDEX
        np.testing.assert_array_equal(host_u16(ws), np.ones(10, np.uint16))


def test_binding_rejects_bad_chains():
    dev = _dev()
    ws = torch.zeros(10, dtype=torch.int16, device=dev)
    with pulse.Plan([pulse.TensorSlot(10, w=ws)]) as plan:
        with pytest.raises(ValueError):
            plan.apply_chain([])
        with pytest.raises(ValueError):
            plan.apply_chain([[]])
        small = torch.zeros(3, dtype=torch.int32, device=dev)
        with pytest.raises(ValueError):
            plan.apply_chain([[(small, torch.zeros(3, dtype=torch.int16, device=dev), 5)]])


def test_prepared_chain_reused():
    """A chain marshalled once and applied twice from the same start gives
    the same result as the oracle both times."""
    dev = _dev()
    rng = np.random.default_rng(41)
    n = 2 * CHUNK + 9
    w0, patches, last = _encode_chain(rng, n, [3e-6, 1e-5])
    w = dev_u16(w0, dev)
    refs = [[_dev_patch(p, dev)] for p in patches]
    with pulse.Plan([pulse.TensorSlot(n, w=w)]) as plan:
        prep = plan.prepare_chain(refs)
        for _ in range(2):
            w.copy_(dev_u16(w0, dev))
            plan.apply_chain(prep)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(host_u16(w), last)
        assert plan.get_error() == 0
        with pulse.Plan([pulse.TensorSlot(n, w=w)]) as other:
            with pytest.raises(ValueError):
                other.apply_chain(prep)


# ------------------------------------------------------------ k-way compose

def _compose(w_sizes, chains, dev, offset=0):
    """GPU k-way composition of chains[t] (per tensor, oldest first); returns
    per tensor (idx, val) of the composed segment and the plan's error word."""
    slots = [pulse.TensorSlot(n, w=torch.zeros(max(n, 1), dtype=torch.int16, device=dev)[:n])
             for n in w_sizes]
    nv = len(chains[0])
    patches = [[_dev_patch(chains[t][v], dev) for t in range(len(w_sizes))] for v in range(nv)]
    # output segments with room for min(n, sum of the versions' counts), guarded
    need = [min(n, sum(chains[t][v][0].size for v in range(nv))) for t, n in enumerate(w_sizes)]
    guards = [(Guarded(max(r, 1), torch.int32, dev), Guarded(max(r, 1), torch.int16, dev))
              for r in need]
    with pulse.Plan(slots) as plan:
        outs, counts = plan.compose_chain(patches, outs=[(gi.t, gv.t) for gi, gv in guards])
        torch.cuda.synchronize()
        err = plan.get_error()
        cnt = counts.cpu().tolist()
        res = [(host_u32_(oi[:k]), host_u16(ov[:k])) for (oi, ov), k in zip(outs, cnt)]
    for gi, gv in guards:
        gi.check("idx_out")
        gv.check("val_out")
    return res, err


def host_u32_(t):
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("nv", [1, 2, 4, 5, 16])
def test_compose_chain_matches_oracle(nv):
    dev = _dev()
    rng = np.random.default_rng(500 + nv)
    etas = ([3e-6, 1e-7, 1e-4, 3e-6, 3e-7] * 4)[:nv]
    chains, finals, w0s = [], [], []
    for n in SIZES:
        w0, patches, last = _encode_chain(rng, n, etas)
        chains.append(patches)
        finals.append(last)
        w0s.append(w0)
    got, err = _compose(SIZES, chains, dev)
    assert err == 0
    for (gi, gv), chain, w0, last in zip(got, chains, w0s, finals):
        oi, ov = oracle.compose_chain(chain)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)
        w = w0.copy()
        oracle.apply(w, gi, gv)
        np.testing.assert_array_equal(w, last)  # one patch brings w0 to the last view


def test_compose_chain_random_overlaps():
    dev = _dev()
    rng = np.random.default_rng(8)
    sizes = [5 * CHUNK + 33, 70000, 9, CHUNK]
    ks = [(4000, 20000, 60000), (30, 2, 0), (9, 9, 1), (CHUNK, CHUNK, CHUNK)]
    chains = [[_rand_patch(rng, n, k) for k in kk] for n, kk in zip(sizes, ks)]
    got, err = _compose(sizes, chains, dev)
    assert err == 0
    for (gi, gv), chain in zip(got, chains):
        oi, ov = oracle.compose_chain(chain)
        np.testing.assert_array_equal(gi, oi)
        np.testing.assert_array_equal(gv, ov)


def test_compose_chain_errors_and_limits():
    dev = _dev()
    n = 3 * CHUNK
    gi = np.arange(0, n, 5, dtype=np.uint32)
    good = (gi, np.ones(gi.size, np.uint16))
    bad_idx = gi.copy()
    bad_idx[10] = n - 1
    _, err = _compose([n], [[good, (bad_idx, good[1])]], dev)
    assert err == pulse.pulse.PULSE_ERR_INDEX
    w = torch.zeros(10, dtype=torch.int16, device=dev)
    with pulse.Plan([pulse.TensorSlot(10, w=w)]) as plan:
        idx = torch.arange(12, dtype=torch.int32, device=dev)
        val = torch.ones(12, dtype=torch.int16, device=dev)
        outs, counts = plan.compose_chain([[(idx, val, 12)]])
        torch.cuda.synchronize()
        assert plan.get_error() == pulse.pulse.PULSE_ERR_INDEX
        assert counts.cpu().tolist() == [10]
        with pytest.raises(ValueError):   # more than 16 versions
            plan.compose_chain([[(idx, val, 3)]] * 17)
        small = [(torch.zeros(2, dtype=torch.int32, device=dev), torch.zeros(2, dtype=torch.int16, device=dev))]
        with pytest.raises(ValueError):   # no room for the union
            plan.compose_chain([[(idx, val, 5)], [(idx, val, 5)]], outs=small)
