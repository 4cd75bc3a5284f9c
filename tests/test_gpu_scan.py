"""GPU parity of the chunked scan (state handoff between chunks) against the
CPU oracle, on the partitions and lifecycle cases of Mamba Streaming State
That Survives Chunking (Let the full scan define legal chunking; Make reset,
checkpoint, and cancellation observable)."""
import functools

import numpy as np
import pytest

import oracle
import synth
from tests._helpers import check_close, empty_like_out, to_device, to_host

pytestmark = pytest.mark.gpu

SEED0 = synth.BASE_SEED + 0       # tiny fp32 shape
SEED1 = synth.BASE_SEED + 1000    # 130M-shaped prefill
SEED4 = synth.BASE_SEED + 4000    # 2.7B-shaped varlen prefill


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


class Scanner:
    """GPU pool + per-slot chunk counters; scans packed chunks of several slots."""

    def __init__(self, m, H, P, N, G, dt_in, dt_dt, n_slots, A, D):
        import torch
        self.m, self.H, self.P, self.N, self.G = m, H, P, N, G
        self.dt_in, self.dt_dt = dt_in, dt_dt
        self.pool = m.ssm_state_init(m.make_config(H, P, N, G, dt_in, dt_dt, 0, 16, 1), n_slots)
        self.seq = np.zeros(n_slots, np.int64)
        self.A, self.D = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()

    def scan(self, slots, chunks, chunk_seq=None):
        """chunks[i] = (x, dt, B, C) numpy of slot slots[i]; returns (status, [y_i numpy])."""
        lens = [c[0].shape[0] for c in chunks]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        cs = [self.seq[s] for s in slots] if chunk_seq is None else chunk_seq
        total = int(cu[-1])
        if total:
            cat = [np.concatenate([c[k] for c in chunks]) for k in range(4)]
            dev = (to_device(cat[0], self.dt_in), to_device(cat[1], self.dt_dt), to_device(cat[2], self.dt_in),
                   to_device(cat[3], self.dt_in))
            y = empty_like_out((total, self.H, self.P), self.dt_in)
        else:
            dev, y = (None,) * 4, None
        st = self.m.ssm_scan_chunk(self.pool, cu, slots, cs, *dev, self.A, self.D, y)
        if st != self.m.SSM_OK:
            return st, None
        for s in slots:
            self.seq[s] += 1
        yh = to_host(y) if total else np.zeros((0, self.H, self.P))
        return st, [yh[cu[i]:cu[i + 1]] for i in range(len(slots))]

    def state(self, slots):
        import torch
        got = torch.empty((len(slots), self.H, self.P, self.N), dtype=torch.float32, device="cuda")
        assert self.m.ssm_state_gather(self.pool, slots, got) == self.m.SSM_OK
        return to_host(got)

    def reset(self, slots):
        assert self.m.ssm_state_reset(self.pool, slots) == self.m.SSM_OK
        for s in slots:
            self.seq[s] = 0

    def close(self):
        self.m.ssm_state_destroy(self.pool)


def _cfg0():
    H, P, N, G, L = 2, 16, 16, 1, 64
    A, D = synth.head_params(SEED0, H)
    x, dt, B, C = synth.tokens(SEED0, 0, L, H, P, G, N)
    return (H, P, N, G, L), A, D, (x, dt, B, C)


def _slice(tok, a, b):
    return tuple(t[a:b] for t in tok)


def _oracle_scan(A, D, tok, dt_in, dt_dt, h0):
    """(y, final state, condition scale of y) of one sequence from h0."""
    st = np.array(h0, np.float64, copy=True)
    y, cond = oracle.scan(st, synth.widen(tok[0], dt_in), synth.widen(tok[1], dt_dt), synth.widen(tok[2], dt_in),
                          synth.widen(tok[3], dt_in), A, D, want_cond=True)
    return y, st, cond


def test_config0_every_listed_partition():
    m = _mod()
    (H, P, N, G, L), A, D, tok = _cfg0()
    y_ref, s_ref, c_ref = _oracle_scan(A, D, tok, synth.F32, synth.F32, np.zeros((H, P, N)))
    parts_list = [[L], [1] * L, [0, L], [32, 0, 32], [7, 13, 43, 1], [L, 0], [63, 1], [2, 3, 5, 7, 11, 13, 17, 6]]
    sc = Scanner(m, H, P, N, G, synth.F32, synth.F32, len(parts_list), A, D)
    try:
        for slot, parts in enumerate(parts_list):
            ys, a = [], 0
            for q in parts:
                st, y = sc.scan([slot], [_slice(tok, a, a + q)])
                assert st == m.SSM_OK
                ys.append(y[0])
                a += q
            check_close(np.concatenate(ys), y_ref, synth.F32, f"y {parts}", positions_axis=0, cond=c_ref)
            check_close(sc.state([slot])[0], s_ref, synth.F32, f"state {parts}")
            _, meta = m.ssm_slot_info(sc.pool, slot)
            assert meta.position == L and meta.next_chunk == len(parts)
        assert m.ssm_pool_status(sc.pool)[1] == 0
    finally:
        sc.close()


def test_config0_reset_swap_duplicate():
    m = _mod()
    (H, P, N, G, L), A, D, tok = _cfg0()
    sc = Scanner(m, H, P, N, G, synth.F32, synth.F32, 4, A, D)
    try:
        # prefix A, reset, B  ==  B from a fresh slot;  and != A then B
        assert sc.scan([0], [_slice(tok, 0, 24)])[0] == m.SSM_OK
        sc.reset([0])
        _, yb_reset = sc.scan([0], [_slice(tok, 24, L)])
        _, yb_fresh = sc.scan([1], [_slice(tok, 24, L)])
        assert np.array_equal(yb_reset[0], yb_fresh[0])
        assert np.array_equal(sc.state([0]), sc.state([1]))
        _, yab = sc.scan([2], [_slice(tok, 0, 24)])
        _, yab2 = sc.scan([2], [_slice(tok, 24, L)])
        assert np.abs(yab2[0] - yb_fresh[0]).max() > 1e-3
        yb_ref, _, yb_cond = _oracle_scan(A, D, _slice(tok, 24, L), synth.F32, synth.F32, np.zeros((H, P, N)))
        check_close(yb_reset[0], yb_ref, synth.F32, "B after reset", cond=yb_cond)
        assert m.ssm_slot_info(sc.pool, 0)[1].epoch == 1
        # swapped chunk order gives a different sequence
        _, y1 = sc.scan([3], [_slice(tok, 24, L)])
        _, y2 = sc.scan([3], [_slice(tok, 0, 24)])
        assert np.abs(y2[0] - yab[0]).max() > 1e-3
        # a chunk number already applied, and a gap: declared, nothing advances
        before = sc.state([2]).copy()
        pos = m.ssm_slot_info(sc.pool, 2)[1].position
        assert sc.scan([2], [_slice(tok, 0, 5)], chunk_seq=[1])[0] == m.SSM_ERR_DUPLICATE
        assert sc.scan([2], [_slice(tok, 0, 5)], chunk_seq=[3])[0] == m.SSM_ERR_SEQUENCE
        assert np.array_equal(sc.state([2]), before) and m.ssm_slot_info(sc.pool, 2)[1].position == pos
        # a multi-sequence call where one slot is out of order advances none of them
        assert sc.scan([1, 2], [_slice(tok, 0, 5), _slice(tok, 0, 5)], chunk_seq=[1, 1])[0] == m.SSM_ERR_DUPLICATE
        assert m.ssm_slot_info(sc.pool, 1)[1].next_chunk == 1
        # released slots refuse
        assert m.ssm_state_release(sc.pool, [3]) == m.SSM_OK
        assert sc.scan([3], [_slice(tok, 0, 5)])[0] == m.SSM_ERR_INVALID_STATE
    finally:
        sc.close()


def test_nonfinite_chunk_poisons_slot_and_leaves_state():
    m = _mod()
    (H, P, N, G, L), A, D, tok = _cfg0()
    sc = Scanner(m, H, P, N, G, synth.F32, synth.F32, 3, A, D)
    try:
        assert sc.scan([0, 1], [_slice(tok, 0, 10), _slice(tok, 0, 10)])[0] == m.SSM_OK
        before = sc.state([0])
        # a NaN in B (shared by every head of the group): no head advances
        bad = [t.copy() for t in _slice(tok, 10, 20)]
        bad[2][4, 0, 3] = np.nan
        assert sc.scan([0, 1], [tuple(bad), _slice(tok, 10, 20)])[0] == m.SSM_OK  # found on the device
        st, flags = m.ssm_pool_status(sc.pool, clear=True)
        assert flags & m.SSM_FLAG_NONFINITE_INPUT
        assert np.array_equal(sc.state([0]), before)            # nothing advanced
        meta0, meta1 = m.ssm_slot_info(sc.pool, 0)[1], m.ssm_slot_info(sc.pool, 1)[1]
        assert meta0.flags & 1 and meta0.position == 10
        assert meta1.flags == 0 and meta1.position == 20        # the healthy sequence went on
        # a NaN in one head's x: that head's state is kept and the slot poisoned
        sc.reset([2])
        assert sc.scan([2], [_slice(tok, 0, 10)])[0] == m.SSM_OK
        keep = sc.state([2])
        bad = [t.copy() for t in _slice(tok, 10, 20)]
        bad[0][4, 1, 3] = np.inf
        assert sc.scan([2], [tuple(bad)])[0] == m.SSM_OK
        assert m.ssm_pool_status(sc.pool, clear=True)[1] & m.SSM_FLAG_NONFINITE_INPUT
        assert np.array_equal(sc.state([2])[0, 1], keep[0, 1])
        assert m.ssm_slot_info(sc.pool, 2)[1].flags & 1
        # a poisoned slot is skipped until reset
        assert sc.scan([0], [_slice(tok, 20, 30)])[0] == m.SSM_OK
        assert m.ssm_pool_status(sc.pool, clear=True)[1] & m.SSM_FLAG_POISONED_SLOT
        assert np.array_equal(sc.state([0]), before)
        sc.reset([0])
        assert m.ssm_slot_info(sc.pool, 0)[1].flags == 0
        assert sc.scan([0], [_slice(tok, 0, 10)])[0] == m.SSM_OK
        assert m.ssm_pool_status(sc.pool)[1] == 0
    finally:
        sc.close()


def test_config1_130m_prefill_chunked_and_partitioned():
    """Mamba-2-130M-shaped layer: d_inner 1536 (24 heads of 64), dstate 128,
    one group, 8 sequences of 2048 bf16 tokens.  Full scan in one call, user
    chunks of 256 with handoff, and seeded random partitions per sequence;
    every sequence and head is checked against the oracle, and the three ways
    of cutting it against each other (at twice the bound, against the
    oracle's condition scale)."""
    m = _mod()
    H, P, N, G, Bt, L = 24, 64, 128, 1, 8, 2048
    A, D = synth.head_params(SEED1, H)
    toks = [synth.tokens(SEED1, b, L, H, P, G, N, synth.BF16, synth.BF16) for b in range(Bt)]
    refs = {b: _oracle_scan(A, D, toks[b], synth.BF16, synth.BF16, np.zeros((H, P, N))) for b in range(Bt)}
    sc = Scanner(m, H, P, N, G, synth.BF16, synth.BF16, 3 * Bt, A, D)
    try:
        # full-sequence scan of all 8 sequences in one call
        st, ys_full = sc.scan(list(range(Bt)), toks)
        assert st == m.SSM_OK
        s_full = sc.state(list(range(Bt)))
        for b in range(Bt):
            check_close(ys_full[b], refs[b][0], synth.BF16, f"full y seq {b}", positions_axis=0, cond=refs[b][2])
            check_close(s_full[b], refs[b][1], synth.BF16, f"full state seq {b}")
        # user chunks of 256 tokens: one call per chunk, all sequences packed
        slots = list(range(Bt, 2 * Bt))
        ys = [[] for _ in range(Bt)]
        for a in range(0, L, 256):
            st, yc = sc.scan(slots, [_slice(t, a, a + 256) for t in toks])
            assert st == m.SSM_OK
            for b in range(Bt):
                ys[b].append(yc[b])
        s_chunk = sc.state(slots)
        for b in range(Bt):
            check_close(np.concatenate(ys[b]), refs[b][0], synth.BF16, f"chunk-256 seq {b}", positions_axis=0,
                        cond=refs[b][2])
            check_close(s_chunk[b], refs[b][1], synth.BF16, f"chunk-256 state seq {b}")
            check_close(np.concatenate(ys[b]), ys_full[b], synth.BF16, f"chunk-256 vs full seq {b}", pair=True,
                        cond=refs[b][2])
            check_close(s_chunk[b], s_full[b], synth.BF16, f"chunk-256 state seq {b}", pair=True)
        # seeded random partitions (with empty chunks) per sequence
        for b in range(Bt):
            parts = synth.random_partition(SEED1, b, L, max_parts=9)
            slot = 2 * Bt + b
            out, a = [], 0
            for q in parts:
                st, yc = sc.scan([slot], [_slice(toks[b], a, a + q)])
                assert st == m.SSM_OK
                out.append(yc[0])
                a += q
            check_close(np.concatenate(out), refs[b][0], synth.BF16, f"partition {parts} seq {b}", cond=refs[b][2])
            check_close(sc.state([slot])[0], refs[b][1], synth.BF16, f"partition state seq {b}")
            check_close(np.concatenate(out), ys_full[b], synth.BF16, f"partition {parts} vs full seq {b}", pair=True,
                        cond=refs[b][2])
            check_close(sc.state([slot])[0], s_full[b], synth.BF16, f"partition state vs full seq {b}", pair=True)
        assert m.ssm_pool_status(sc.pool)[1] == 0
    finally:
        sc.close()


@functools.lru_cache(maxsize=2)
def _config4_wave(wave):
    """Tokens of the 64 sequences of one wave of the 2.7B-shaped varlen workload."""
    H, P, N, G, S = 80, 64, 128, 1, 64
    lens = synth.varlen_lengths(SEED4, S, 512, 8192)
    return tuple(synth.tokens(SEED4, 1000 * wave + i, int(lens[i]), H, P, G, N, synth.BF16, synth.BF16)
                 for i in range(S))


@pytest.mark.parametrize("chunk", [256, 1024])
def test_config4_varlen_packed_with_slot_reuse(chunk):
    """Mamba-2-2.7B-shaped layer: d_inner 5120 (80 heads of 64), dstate 128,
    one group; 64 packed sequences with lengths U(512, 8192) fed as user
    chunks of 256 or 1024 tokens (every call packs the next chunk of each live
    sequence).  Then the 64 slots are reset and reused by a second wave,
    each checked against a fresh-state scan; a control wave without the
    reset must differ."""
    m = _mod()
    H, P, N, G, S = 80, 64, 128, 1, 64
    A, D = synth.head_params(SEED4, H)
    lens = synth.varlen_lengths(SEED4, S, 512, 8192)
    sc = Scanner(m, H, P, N, G, synth.BF16, synth.BF16, 2 * S, A, D)
    heads = [0, 41, 79]
    try:
        for wave in range(2):
            toks = list(_config4_wave(wave))
            if wave == 1:
                sc.reset(list(range(S)))
            ys = [[] for _ in range(S)]
            for a in range(0, int(lens.max()), chunk):
                live = [i for i in range(S) if lens[i] > a]
                st, yc = sc.scan(live, [_slice(toks[i], a, min(a + chunk, int(lens[i]))) for i in live])
                assert st == m.SSM_OK
                for i, y in zip(live, yc):
                    ys[i].append(y)
            states = sc.state(list(range(S)))
            for i in (0, 17, 63):
                y_all = np.concatenate(ys[i])
                assert y_all.shape[0] == lens[i]
                for h in heads:
                    t = toks[i]
                    st0 = np.zeros((P, N))
                    yo, yc = oracle.scan_head(st0, synth.widen(t[0][:, h], synth.BF16),
                                              synth.widen(t[1][:, h], synth.BF16), synth.widen(t[2][:, 0], synth.BF16),
                                              synth.widen(t[3][:, 0], synth.BF16), A[h], D[h], want_cond=True)
                    check_close(y_all[:, h], yo, synth.BF16, f"chunk {chunk} wave {wave} seq {i} head {h}",
                                positions_axis=0, cond=yc)
                    check_close(states[i, h], st0, synth.BF16, f"wave {wave} seq {i} head {h} state")
            if wave == 1:
                # control: wave-2 tokens of sequence 0 on a slot still holding
                # wave-1's final state (no reset) must give different outputs
                first = synth.tokens(SEED4, 0, int(lens[0]), H, P, G, N, synth.BF16, synth.BF16)
                assert sc.scan([S], [first])[0] == m.SSM_OK
                _, yc = sc.scan([S], [_slice(toks[0], 0, 256)])
                assert np.abs(yc[0] - ys[0][0][:256]).max() > 1e-2
        assert m.ssm_pool_status(sc.pool)[1] == 0
    finally:
        sc.close()


# head counts and groups of the tensor-core scan cases: two groups of two heads, one group of three
KERNELS = [(4, 2, "scan_ssd"), (3, 1, "scan_ssd")]


@pytest.mark.parametrize("H,G,path", KERNELS)
@pytest.mark.parametrize("lens,dt_dt", [([1, 5, 127, 128, 129, 300], synth.F32), ([0, 64, 256, 383], synth.BF16)])
def test_tensor_core_scan_ragged_lengths(lens, dt_dt, H, G, path):
    """The tensor-core chunked scan (bf16 x/B/C, headdim 64, dstate 128) on
    lengths around its 128-token kernel chunk, then a second call that
    continues every sequence from its handed-off state."""
    m = _mod()
    P, N = 64, 128
    seed = SEED1 + 77
    A, D = synth.head_params(seed, H)
    S = len(lens)
    sc = Scanner(m, H, P, N, G, synth.BF16, dt_dt, S, A, D)
    try:
        states = [np.zeros((H, P, N)) for _ in range(S)]
        for call in range(2):
            toks = [synth.tokens(seed, 100 * call + i, L, H, P, G, N, synth.BF16, dt_dt) for i, L in enumerate(lens)]
            st, ys = sc.scan(list(range(S)), toks)
            assert st == m.SSM_OK
            if any(lens):
                assert m.ssm_last_path(sc.pool) == path
            got = sc.state(list(range(S)))
            for i in range(S):
                y_ref, states[i], y_cond = _oracle_scan(A, D, toks[i], synth.BF16, dt_dt, states[i])
                check_close(ys[i], y_ref, synth.BF16, f"call {call} seq {i} (L={lens[i]}) y", positions_axis=0,
                            cond=y_cond)
                check_close(got[i], states[i], synth.BF16, f"call {call} seq {i} state")
            assert m.ssm_pool_status(sc.pool)[1] == 0
    finally:
        sc.close()


@pytest.mark.parametrize("H,G,path", KERNELS)
def test_tensor_core_scan_fast_decay_takes_the_exact_form(H, G, path):
    """The tensor-core scan factors exp(cum_i - cum_j) around a reference
    point of each 128-token chunk only while both factors stay far inside
    fp32; where the decay over the chunk is steeper (here heads with A = -40
    and -400, and a stretch of one sequence with 30 times larger dt) the
    two-head kernel cuts the chunk into shorter passes and the one-head
    kernel takes its exact per-block form.  Mixed within one sequence and
    across its calls, they match the oracle."""
    m = _mod()
    P, N = 64, 128
    seed = SEED1 + 79
    _, D = synth.head_params(seed, H)
    A = np.array([-1.0, -3.0, -40.0, -400.0][-H:], np.float32)
    lens = [300, 129, 384]
    S = len(lens)
    sc = Scanner(m, H, P, N, G, synth.BF16, synth.F32, S, A, D)
    try:
        states = [np.zeros((H, P, N)) for _ in range(S)]
        for call in range(2):
            toks = [list(synth.tokens(seed, 100 * call + i, L, H, P, G, N, synth.BF16, synth.F32))
                    for i, L in enumerate(lens)]
            toks[0][1] = toks[0][1].copy()
            toks[0][1][150:260] *= np.float32(30.0)   # dt: a steep stretch in the middle of sequence 0
            toks = [tuple(t) for t in toks]
            st, ys = sc.scan(list(range(S)), toks)
            assert st == m.SSM_OK and m.ssm_last_path(sc.pool) == path
            got = sc.state(list(range(S)))
            for i in range(S):
                y_ref, states[i], y_cond = _oracle_scan(A, D, toks[i], synth.BF16, synth.F32, states[i])
                check_close(ys[i], y_ref, synth.BF16, f"call {call} seq {i} y", positions_axis=0, cond=y_cond)
                check_close(got[i], states[i], synth.BF16, f"call {call} seq {i} state")
            assert m.ssm_pool_status(sc.pool)[1] == 0
    finally:
        sc.close()


@pytest.mark.parametrize("H,G,path", KERNELS)
@pytest.mark.parametrize("where", ["B", "C", "x", "dt"])
def test_tensor_core_scan_nonfinite_poisons_slot(where, H, G, path):
    """bf16 scan on the tensor cores: a NaN or Inf in a sequence's B, C, x or
    dt flags SSM_FLAG_NONFINITE_INPUT, poisons its slot and leaves the state
    of every head it reaches as it was; the other sequence of the call
    advances and matches the oracle."""
    m = _mod()
    P, N = 64, 128
    seed = SEED1 + 91
    A, D = synth.head_params(seed, H)
    sc = Scanner(m, H, P, N, G, synth.BF16, synth.F32, 2, A, D)
    try:
        toks = [synth.tokens(seed, i, 300, H, P, G, N, synth.BF16, synth.F32) for i in range(2)]
        assert sc.scan([0, 1], [_slice(t, 0, 150) for t in toks])[0] == m.SSM_OK
        assert m.ssm_last_path(sc.pool) == path
        before = sc.state([0, 1])
        bad = [t.copy() for t in _slice(toks[0], 150, 300)]
        nan16, inf16 = np.uint16(0x7FC0), np.uint16(0x7F80)  # bf16 bit patterns
        if where == "B":
            bad[2][140, 0, 5] = nan16      # group 0: heads 0 and 1 (and 2 with one group)
        elif where == "C":
            bad[3][140, 0, 5] = inf16
        elif where == "x":
            bad[0][140, 1, 7] = inf16      # head 1
        else:
            bad[1][140, 1] = np.nan
        assert sc.scan([0, 1], [tuple(bad), _slice(toks[1], 150, 300)])[0] == m.SSM_OK  # found on the device
        assert m.ssm_last_path(sc.pool) == path
        assert m.ssm_pool_status(sc.pool, clear=True)[1] & m.SSM_FLAG_NONFINITE_INPUT
        after = sc.state([0, 1])
        for h in ([0, 1] if where in ("B", "C") else [1]):
            assert np.array_equal(after[0, h], before[0, h]), h
        meta0 = m.ssm_slot_info(sc.pool, 0)[1]
        assert meta0.flags & 1
        if where in ("B", "C"):
            assert meta0.position == 150
        _, ref, _ = _oracle_scan(A, D, toks[1], synth.BF16, synth.F32, np.zeros((H, P, N)))
        check_close(after[1], ref, synth.BF16, "the healthy sequence's state")
        assert m.ssm_slot_info(sc.pool, 1)[1].flags == 0
    finally:
        sc.close()
