"""Benchmark of the Mamba-2 state-update hot path on GB300.

Headline metric: batched decode state-update throughput (tokens/s) and the
HBM bandwidth it achieves, on the Nemotron-shaped decode workload: 256
requests, 128 heads of headdim 64, dstate 128, 8 groups, bf16 x/B/C, fp32
dt, fp32 state (4 MiB per request).  One benchmark step is one pass of that
workload: 64 successive single-token decode steps of all 256 requests
(16384 tokens, 64 kernel launches).

Also measured in the same run, each in its own timed region:
  * speculative verify at batch 512 (same head shape, T = 8 drafts,
    acceptance 0.8, window 16): copy flavour and ReplaySSM flavour, verify +
    commit per step, over 32 verify steps, next to a plain decode step at
    batch 512;
  * chunked prefill scan of 8 sequences x 2048 tokens (Mamba-2-130M-shaped
    layer: 24 heads of 64, dstate 128, bf16);
  * launch cost at small batch: decode (batch 1, 8, 64) and replay verify +
    commit (batch 8) issued call by call and as a replayed CUDA graph, with
    the capture's own cost;
  * a gated-delta-rule layer (32 value heads, 16 key heads, 128 x 128 state
    per head, batch 256): in-place decode, the replay pool used for plain
    decode, and replay verify + commit with 8 drafts;
  * the oracle (CPU, fp64) on a bounded sample of the decode workload.

Inputs are seeded synthetic data drawn on the device (x, B, C ~ N(0,1),
dt = softplus(N(-2, 0.5)), A = -exp(U(0, 1.5)), D ~ N(0, 1), state
N(0, 0.1)); the state (1 GiB) is larger than L2, so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica on its own GPU (the
recurrence has no cross-request exchange); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SEED = 20261202 + 2000

# decode workload (Nemotron-shaped heads)
DEC = dict(H=128, P=64, N=128, G=8, R=256, tokens=64)
# speculative verify workload
VER = dict(H=128, P=64, N=128, G=8, R=512, T=8, p=0.8, W=16, steps=32)
# prefill workload (Mamba-2-130M-shaped layer)
PRE = dict(H=24, P=64, N=128, G=1, R=8, L=2048)
# gated delta rule layer: 32 value heads, 16 key heads, 128 x 128 fp32 state per head (2 MiB a request)
GDN = dict(H=32, G=16, dk=128, dv=128, R=256, tokens=64, T=8, p=0.8, W=16, steps=32)


def algorithmic_bytes_decode(R, H, P, N, G, in_b=2):
    """State read + write, token inputs (x, dt, B, C) and output y, per step."""
    state = 2 * R * H * P * N * 4
    inputs = R * (H * P * in_b + H * 4 + 2 * G * N * in_b)
    out = R * H * P * in_b
    return state + inputs + out


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1882.2)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _file_hash(*paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_name, *sources):
    """DRAM bytes per launch recorded in a profiles/ summary, if the kernel
    source it was taken from is unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m_t or not m_h:
        return None
    if m_h.group(1) != _file_hash(*[os.path.join(ROOT, s) for s in sources]):
        return None
    return float(m_t.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        rows = [r for r in open(self.out.name).read().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            f = [c.strip() for c in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# synthetic inputs on the device

def _gen(torch, shape, gen, dtype, kind):
    if kind == "normal":
        t = torch.randn(shape, generator=gen, device="cuda", dtype=torch.float32)
    elif kind == "dt":
        t = torch.nn.functional.softplus(torch.randn(shape, generator=gen, device="cuda") * 0.5 - 2.0)
    else:
        raise ValueError(kind)
    return t.to(dtype).contiguous()


def step_inputs(torch, gen, n, H, P, G, N, n_tok=None):
    lead = (n,) if n_tok is None else (n, n_tok)
    return (_gen(torch, lead + (H, P), gen, torch.bfloat16, "normal"),
            _gen(torch, lead + (H,), gen, torch.float32, "dt"),
            _gen(torch, lead + (G, N), gen, torch.bfloat16, "normal"),
            _gen(torch, lead + (G, N), gen, torch.bfloat16, "normal"))


def head_params(torch, gen, H):
    A = -torch.exp(torch.rand(H, generator=gen, device="cuda") * 1.5)
    D = torch.randn(H, generator=gen, device="cuda")
    return A.contiguous(), D.contiguous()


# ---------------------------------------------------------------------------
# the measured workloads

def bench_decode(torch, m, dist, args, clocks):
    c = DEC
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 17 * args.rank)
    H, P, N, G, R, T = c["H"], c["P"], c["N"], c["G"], c["R"], c["tokens"]
    A, D = head_params(torch, gen, H)
    init = (torch.randn((R, H, P, N), generator=gen, device="cuda") * 0.1).contiguous()
    pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_F32, m.SSM_MODE_COPY, 16, 1),
                            R, init)
    del init
    x, dt, B, C = step_inputs(torch, gen, T * R, H, P, G, N)
    x, dt, B, C = (t.view(T, R, *t.shape[1:]) for t in (x, dt, B, C))
    y = torch.empty((T, R, H, P), dtype=torch.bfloat16, device="cuda")
    slots = list(range(R))
    stream = torch.cuda.current_stream()

    def one_step():  # 64 successive decode tokens of all requests
        for t in range(T):
            st = m.ssm_decode_step(pool, slots, x[t], dt[t], B[t], C[t], A, D, y[t], stream=stream)
            if st != m.SSM_OK:
                raise m.SSMError(st, "ssm_decode_step")

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    # per-launch durations of the decode kernel, for the roofline
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(T)]
    for t in range(T):
        ev[t][0].record(stream)
        m.ssm_decode_step(pool, slots, x[t], dt[t], B[t], C[t], A, D, y[t], stream=stream)
        ev[t][1].record(stream)
    torch.cuda.synchronize()
    launch_ms = [a.elapsed_time(b) for a, b in ev]

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        one_step()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    st, flags = m.ssm_pool_status(pool)
    assert st == m.SSM_OK and flags == 0, f"decode raised device flags {flags}"
    m.ssm_state_destroy(pool)
    return dict(ms=ms, launch_ms=statistics.median(launch_ms), launch_mean_ms=sum(launch_ms) / T,
                tokens=R * T * args.steps, launches=T * args.steps, clocks=clk,
                bytes_per_launch=algorithmic_bytes_decode(R, H, P, N, G))


def bench_decode_e2e(torch, m, args):
    """The same decode workload through the C ABI's host-buffer entry
    (ssm_decode_steps_host): every token's inputs go up from pinned host
    memory and its output comes back inside the timed region, the library
    overlapping token t + 1's upload and token t - 1's readback with token t's
    decode on its own copy streams."""
    c = DEC
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 91 + 17 * args.rank)
    H, P, N, G, R, T = c["H"], c["P"], c["N"], c["G"], c["R"], c["tokens"]
    A, D = head_params(torch, gen, H)
    init = (torch.randn((R, H, P, N), generator=gen, device="cuda") * 0.1).contiguous()
    pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_F32, m.SSM_MODE_COPY, 16, 1),
                            R, init)
    del init
    dev_in = step_inputs(torch, gen, T * R, H, P, G, N)
    host_in = [t.cpu().pin_memory() for t in dev_in]
    del dev_in
    y_host = torch.empty((T, R, H, P), dtype=torch.bfloat16).pin_memory()
    slots = list(range(R))
    stream = torch.cuda.current_stream()

    def one_step():
        st = m.ssm_decode_steps_host(pool, slots, T, *host_in, A, D, y_host, stream=stream)
        assert st == m.SSM_OK, f"ssm_decode_steps_host returned {st}"

    for _ in range(max(1, args.warmup)):
        one_step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        one_step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    st, flags = m.ssm_pool_status(pool)
    assert st == m.SSM_OK and flags == 0, f"host-buffer decode raised device flags {flags}"
    m.ssm_state_destroy(pool)
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = y_host.numel() * y_host.element_size()
    return dict(ms=ms, tokens=R * T * args.steps, h2d=h2d, d2h=d2h)


def _verify_bytes(acc_np, R, H, P, N, G, T1, W, S, warm):
    """Algorithmic bytes per step of copy and replay verify (+ commit).
    Copy: read the state, write T+1 states, token inputs and outputs.  Replay:
    read the checkpoint and the k logged entries, token inputs and outputs,
    stage the step's entries after the log; a fold reads the checkpoint and
    its m entries and writes the checkpoint.  Log lengths and folds follow the
    commit rule on the same accept counts (integer bookkeeping only), warm-up
    steps included so the timed steps start from the logs they leave."""
    state = H * P * N * 4
    tok_in = H * P * 2 + H * 4 + 2 * G * N * 2
    entry = H * P * 2 + H * 4 + G * N * 2
    y_b = H * P * 2
    copy_b = R * (state * (T1 + 1) + T1 * (tok_in + y_b))
    total, folds = 0, 0
    k = [0] * R
    for n_run, counted in ((warm, False), (S, True)):
        for step in range(n_run):
            for r in range(R):
                kept = int(acc_np[step % S][r]) + 1
                b = state + k[r] * entry + T1 * (tok_in + y_b + entry)
                if k[r] + kept >= W:
                    b += 2 * state + (k[r] + kept) * entry
                    k[r] = 0
                    folds += counted
                else:
                    k[r] += kept
                if counted:
                    total += b
    return copy_b, total / S, folds / S


def _verify_bytes_fold_in_verify(acc_np, R, H, P, N, G, T1, W, S, warm):
    """Algorithmic bytes per step of replay verify (+ commit) when the verify
    folds a full log: read the checkpoint and the k logged entries, token
    inputs and outputs, stage the step's entries; a request whose log holds W
    or more tokens also writes its new checkpoint (its log was read above).
    The commit only appends.  Log lengths follow that rule on the same accept
    counts, warm-up steps included."""
    state = H * P * N * 4
    tok_in = H * P * 2 + H * 4 + 2 * G * N * 2
    entry = H * P * 2 + H * 4 + G * N * 2
    y_b = H * P * 2
    total, folds = 0, 0
    k = [0] * R
    for n_run, counted in ((warm, False), (S, True)):
        for step in range(n_run):
            for r in range(R):
                b = state + k[r] * entry + T1 * (tok_in + y_b + entry)
                if k[r] >= W:
                    b += state
                    k[r] = 0
                    folds += counted
                k[r] += int(acc_np[step % S][r]) + 1
                if counted:
                    total += b
    return total / S, folds / S


def bench_verify(torch, m, args, T=None, p=None, windows=None, static=False):
    """Copy verify vs ReplaySSM verify at batch 512, verify + commit per step,
    at one (T, p) and the given windows (the copy flavour does not depend on
    the window).  With static, also the replay verify through the entry point
    that allocates nothing, on caller-owned checkpoint and log buffers."""
    import synth
    c = VER
    H, P, N, G, R, S = c["H"], c["P"], c["N"], c["G"], c["R"], c["steps"]
    T = c["T"] if T is None else T
    p = c["p"] if p is None else p
    windows = [c["W"]] if windows is None else list(windows)
    T1 = T + 1
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 33 + 17 * args.rank)
    A, D = head_params(torch, gen, H)
    acc = torch.from_numpy(synth.accept_counts(SEED, S, R, T, p)).cuda()
    acc_np = acc.cpu().numpy()
    n_sets = 4  # distinct step inputs, cycled
    ins = [step_inputs(torch, gen, R, H, P, G, N, n_tok=T1) for _ in range(n_sets)]
    y = torch.empty((R, T1, H, P), dtype=torch.bfloat16, device="cuda")
    slots = list(range(R))
    stream = torch.cuda.current_stream()
    peak, _, kind = measured_peaks()
    warm = 3
    out = {"replay": {}, "replay_fold_in_verify": {}}
    runs = ([(m.SSM_MODE_COPY, "copy", windows[0], m.SSM_FOLD_AT_COMMIT)] +
            [(m.SSM_MODE_REPLAY, "replay", W, m.SSM_FOLD_AT_COMMIT) for W in windows] +
            [(m.SSM_MODE_REPLAY, "replay_fold_in_verify", W, m.SSM_FOLD_IN_VERIFY) for W in windows])
    for mode, name, W, fold in runs:
        init = (torch.randn((R, H, P, N), generator=gen, device="cuda") * 0.1).contiguous()
        pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_F32, mode, W, T1,
                                              fold=fold), R, init)
        del init
        verify = m.ssm_verify_copy if mode == m.SSM_MODE_COPY else m.ssm_verify_replay

        def run(n_steps):
            for s in range(n_steps):
                x, dt, B, C = ins[s % n_sets]
                verify(pool, slots, T1, x, dt, B, C, A, D, y, stream=stream)
                m.ssm_state_commit(pool, slots, acc[s % S], False, A, stream=stream)

        run(warm)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(S)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        paths = m.ssm_last_path(pool)
        st, flags = m.ssm_pool_status(pool)
        assert st == m.SSM_OK and flags == 0, f"{name} verify raised device flags {flags}"
        copy_b, replay_b, folds = _verify_bytes(acc_np, R, H, P, N, G, T1, W, S, warm)
        if fold == m.SSM_FOLD_IN_VERIFY:
            replay_b, folds = _verify_bytes_fold_in_verify(acc_np, R, H, P, N, G, T1, W, S, warm)
        b = copy_b if mode == m.SSM_MODE_COPY else replay_b
        us = 1000.0 * ms / S
        gbs = b / (us * 1e-6) / 1e9
        rec = dict(us_per_step=us, algorithmic_bytes=b, achieved_gbs=gbs, frac_of_hbm=gbs / peak,
                   frac_of_nominal_8tbs=gbs / 8000.0)
        if mode == m.SSM_MODE_COPY:
            out["copy"] = rec
            # plain decode step at the same batch, for the ratios
            xd, dtd, Bd, Cd = (t[:, 0].contiguous() for t in ins[0])
            yd = torch.empty((R, H, P), dtype=torch.bfloat16, device="cuda")
            for _ in range(3):
                m.ssm_decode_step(pool, slots, xd, dtd, Bd, Cd, A, D, yd, stream=stream)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(S):
                m.ssm_decode_step(pool, slots, xd, dtd, Bd, Cd, A, D, yd, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            out["plain_decode_us"] = 1000.0 * e0.elapsed_time(e1) / S
        else:
            rec.update(W=W, folds_per_step=folds, commit_path=paths,
                       over_plain=us / out["plain_decode_us"], copy_over_replay=out["copy"]["us_per_step"] / us)
            if fold == m.SSM_FOLD_IN_VERIFY:
                rec["vs_fold_at_commit"] = out["replay"][str(W)]["us_per_step"] / us
            out[name][str(W)] = rec
        m.ssm_state_destroy(pool)
    if static:
        # the entry point that allocates nothing: verify only (the caller folds), logs of the lengths the
        # commit rule gives mid-run, against the pool's verify alone at the same lengths
        W = windows[0]
        Wc = W - 1 + T1
        ckpt = (torch.randn((R, H, P, N), generator=gen, device="cuda") * 0.1).contiguous()
        log_x = torch.randn((R, Wc, H, P), generator=gen, device="cuda").bfloat16()
        log_dt = torch.full((R, Wc, H), 0.1, device="cuda")
        log_B = torch.randn((R, Wc, G, N), generator=gen, device="cuda").bfloat16()
        log_len = torch.randint(0, W, (R,), generator=gen, device="cuda", dtype=torch.int32)
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")

        def run_static(n):
            for s in range(n):
                x, dt, B, C = ins[s % n_sets]
                assert m.ssm_verify_replay_static(R, T1, H, P, N, G, W, m.SSM_DTYPE_BF16, m.SSM_DTYPE_F32, ckpt,
                                                  log_x, log_dt, log_B, log_len, x, dt, B, C, A, D, y, flags,
                                                  stream=stream) == m.SSM_OK
        run_static(warm)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_static(S)
        e1.record(stream)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        out["static_verify_us"] = 1000.0 * e0.elapsed_time(e1) / S
        out["static_path"] = m.ssm_last_path(None)
        del ckpt, log_x, log_dt, log_B
    out["hbm_peak_source"] = kind
    out["copy_over_plain"] = out["copy"]["us_per_step"] / out["plain_decode_us"]
    out["config"] = dict(batch=R, T=T, p=p, windows=windows, steps=S, heads=H, headdim=P, dstate=N, groups=G)
    return out


def bench_verify_sweep(torch, m, args):
    """Every (T, p, W) point of the speculative verify workload at batch 512:
    T in {4, 8}, p in {0.6, 0.8}, W in {8, 16, 32}; verify + commit per step."""
    pts = []
    for T in (4, 8):
        for p in (0.6, 0.8):
            r = bench_verify(torch, m, args, T=T, p=p, windows=(8, 16, 32))
            for W, rec in r["replay"].items():
                pts.append(dict(T=T, p=p, W=int(W), copy_us=r["copy"]["us_per_step"],
                                copy_frac_of_hbm=r["copy"]["frac_of_hbm"], replay_us=rec["us_per_step"],
                                replay_frac_of_hbm=rec["frac_of_hbm"], replay_frac_of_nominal=rec["frac_of_nominal_8tbs"],
                                folds_per_step=rec["folds_per_step"], copy_over_replay=rec["copy_over_replay"],
                                replay_over_plain=rec["over_plain"], commit_path=rec["commit_path"],
                                fold_in_verify_us=r["replay_fold_in_verify"][W]["us_per_step"],
                                fold_in_verify_frac_of_hbm=r["replay_fold_in_verify"][W]["frac_of_hbm"]))
    return dict(points=pts, config=dict(batch=VER["R"], steps=VER["steps"], heads=VER["H"], headdim=VER["P"],
                                        dstate=VER["N"], groups=VER["G"]))


def bench_prefill(torch, m, args):
    c = PRE
    H, P, N, G, R, L = c["H"], c["P"], c["N"], c["G"], c["R"], c["L"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 55 + 17 * args.rank)
    A, D = head_params(torch, gen, H)
    x = _gen(torch, (R * L, H, P), gen, torch.bfloat16, "normal")
    dt = _gen(torch, (R * L, H), gen, torch.bfloat16, "dt")
    B = _gen(torch, (R * L, G, N), gen, torch.bfloat16, "normal")
    C = _gen(torch, (R * L, G, N), gen, torch.bfloat16, "normal")
    y = torch.empty_like(x)
    pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_BF16, m.SSM_MODE_COPY, 16, 1), R)
    cu = [i * L for i in range(R + 1)]
    slots = list(range(R))
    stream = torch.cuda.current_stream()
    seq = 0

    def run(n):
        nonlocal seq
        for _ in range(n):
            m.ssm_state_reset(pool, slots, stream=stream)
            st = m.ssm_scan_chunk(pool, cu, slots, [0] * R, x, dt, B, C, A, D, y, stream=stream)
            if st != m.SSM_OK:
                raise m.SSMError(st, "ssm_scan_chunk")

    run(2)
    torch.cuda.synchronize()
    n = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(n)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    path = m.ssm_last_path(pool)
    m.ssm_state_destroy(pool)
    alg = 2 * R * L * H * P * 2 + R * L * (H * 2 + 2 * G * N * 2) + R * H * P * N * 4
    # DRAM bytes of one scan from the profile (taken at 16 sequences, traffic in proportion to them)
    prof = profiled_traffic("scan_ssd_kernel_130m.md", "hybrid_serving_mamba_gb300/csrc/scan_ssd.cu",
                            "hybrid_serving_mamba_gb300/csrc/tc.cuh", "hybrid_serving_mamba_gb300/csrc/tma.cuh")
    traffic = prof * R / 16 if prof is not None else None
    return dict(us_per_scan=1000 * ms, tokens_per_s=R * L / (ms / 1000), path=path, traffic=traffic,
                achieved_gbs=alg / (ms / 1000) / 1e9, algorithmic_bytes=alg,
                frac_of_hbm=alg / (ms / 1000) / 1e9 / measured_peaks()[0],
                config=dict(seqs=R, seqlen=L, heads=H, headdim=P, dstate=N, groups=G, includes="reset + scan"))


def bench_prefill_varlen(torch, m, args, chunk=1024, S=64):
    """2.7B-shaped layer (80 heads of 64, dstate 128, one group): S packed
    sequences (64 in the workload) with lengths U(512, 8192), fed as user
    chunks of `chunk` tokens (each call packs the next chunk of every live
    sequence).  Time per wave of all sequences, from reset."""
    import synth
    H, P, N, G = 80, 64, 128, 1
    lens = synth.varlen_lengths(SEED + 4000, S, 512, 8192)
    total = int(lens.sum())
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 77 + 17 * args.rank)
    A, D = head_params(torch, gen, H)
    x = _gen(torch, (total, H, P), gen, torch.bfloat16, "normal")
    dt = _gen(torch, (total, H), gen, torch.bfloat16, "dt")
    B = _gen(torch, (total, G, N), gen, torch.bfloat16, "normal")
    C = _gen(torch, (total, G, N), gen, torch.bfloat16, "normal")
    starts = [0]
    for L in lens[:-1]:
        starts.append(starts[-1] + int(L))
    # pack each call's chunks contiguously (the layout a serving engine hands over)
    calls = []
    for a0 in range(0, int(lens.max()), chunk):
        live = [i for i in range(S) if lens[i] > a0]
        idx = torch.cat([torch.arange(starts[i] + a0, starts[i] + min(a0 + chunk, int(lens[i])), device="cuda")
                         for i in live])
        cu = [0]
        for i in live:
            cu.append(cu[-1] + min(a0 + chunk, int(lens[i])) - a0)
        calls.append((live, cu, x[idx].contiguous(), dt[idx].contiguous(), B[idx].contiguous(), C[idx].contiguous(),
                      torch.empty((len(idx), H, P), dtype=torch.bfloat16, device="cuda")))
    del x, dt, B, C
    pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_BF16, m.SSM_MODE_COPY, 16, 1), S)
    stream = torch.cuda.current_stream()

    def wave():
        m.ssm_state_reset(pool, list(range(S)), stream=stream)
        for q, (live, cu, xc, dc, bc, cc, yc) in enumerate(calls):
            st = m.ssm_scan_chunk(pool, cu, live, [q] * len(live), xc, dc, bc, cc, A, D, yc, stream=stream)
            if st != m.SSM_OK:
                raise m.SSMError(st, "ssm_scan_chunk")

    wave()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 3
    e0.record(stream)
    for _ in range(n):
        wave()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    path = m.ssm_last_path(pool)
    st, flags = m.ssm_pool_status(pool)
    assert st == m.SSM_OK and flags == 0, f"varlen prefill raised device flags {flags}"
    m.ssm_state_destroy(pool)
    alg = 2 * total * H * P * 2 + total * (H * 2 + 2 * G * N * 2) + S * H * P * N * 4
    return dict(ms_per_wave=ms, tokens=total, tokens_per_s=total / (ms / 1000), path=path,
                achieved_gbs=alg / (ms / 1000) / 1e9, algorithmic_bytes=alg, calls_per_wave=len(calls),
                frac_of_hbm=alg / (ms / 1000) / 1e9 / measured_peaks()[0],
                config=dict(seqs=S, lengths="U(512, 8192)", user_chunk=chunk, heads=H, headdim=P, dstate=N,
                            groups=G, includes="reset + every chunk call"))


def bench_replay_plain_decode(torch, m, args):
    """ReplaySSM used for plain decode (one token per step, no drafts): the
    batch-256 decode workload through verify_replay (n_tok = 1) + commit,
    window 16, against the in-place decode step."""
    c = DEC
    H, P, N, G, R, T = c["H"], c["P"], c["N"], c["G"], c["R"], c["tokens"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 131 + 17 * args.rank)
    A, D = head_params(torch, gen, H)
    x, dt, B, C = step_inputs(torch, gen, T * R, H, P, G, N)
    x, dt, B, C = (t.view(T, R, *t.shape[1:]) for t in (x, dt, B, C))
    zeros = torch.zeros(R, dtype=torch.int32, device="cuda")
    y = torch.empty((R, H, P), dtype=torch.bfloat16, device="cuda")
    slots = list(range(R))
    stream = torch.cuda.current_stream()
    out = {}
    for name, mode, fold in (("decode", m.SSM_MODE_COPY, m.SSM_FOLD_AT_COMMIT),
                             ("replay", m.SSM_MODE_REPLAY, m.SSM_FOLD_AT_COMMIT),
                             ("replay_fold_in_verify", m.SSM_MODE_REPLAY, m.SSM_FOLD_IN_VERIFY)):
        init = (torch.randn((R, H, P, N), generator=gen, device="cuda") * 0.1).contiguous()
        pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_F32, mode, 16, 1,
                                              fold=fold), R, init)
        del init

        def run(n):
            for t in range(n):
                k = t % T
                if mode == m.SSM_MODE_COPY:
                    m.ssm_decode_step(pool, slots, x[k], dt[k], B[k], C[k], A, D, y, stream=stream)
                else:
                    m.ssm_verify_replay(pool, slots, 1, x[k], dt[k], B[k], C[k], A, D, y, stream=stream)
                    m.ssm_state_commit(pool, slots, zeros, False, A, stream=stream)

        run(16)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(T)
        e1.record(stream)
        torch.cuda.synchronize()
        out[name + "_us_per_step"] = 1000.0 * e0.elapsed_time(e1) / T
        st, flags = m.ssm_pool_status(pool)
        assert st == m.SSM_OK and flags == 0, f"{name} raised device flags {flags}"
        m.ssm_state_destroy(pool)
    out["replay_speedup_over_decode"] = out["decode_us_per_step"] / out["replay_us_per_step"]
    out["replay_fold_in_verify_speedup_over_decode"] = (out["decode_us_per_step"] /
                                                       out["replay_fold_in_verify_us_per_step"])
    out["config"] = dict(batch=R, W=16, tokens=T, heads=H, headdim=P, dstate=N, groups=G)
    return out


def gdn_inputs(torch, gen, n, H, G, dk, dv, n_tok=None):
    """q, k (unit length per key head), v in bf16; g = log gate and beta in fp32."""
    lead = (n,) if n_tok is None else (n, n_tok)
    q = torch.nn.functional.normalize(torch.randn(lead + (G, dk), generator=gen, device="cuda"), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(lead + (G, dk), generator=gen, device="cuda"), dim=-1)
    v = torch.randn(lead + (H, dv), generator=gen, device="cuda")
    sp = torch.nn.functional.softplus(torch.randn(lead + (H,), generator=gen, device="cuda") * 0.5 - 2.0)
    g = -sp * torch.exp(torch.rand(lead + (H,), generator=gen, device="cuda") * 1.5)
    beta = torch.sigmoid(torch.randn(lead + (H,), generator=gen, device="cuda"))
    return (q.bfloat16().contiguous(), k.bfloat16().contiguous(), v.bfloat16().contiguous(), g.contiguous(),
            beta.contiguous())


def algorithmic_bytes_gdn_decode(R, H, G, dk, dv, in_b=2):
    """State read + write, the token's q, k, v, g, beta and the output y, per step of R requests."""
    return R * (2 * H * dv * dk * 4 + 2 * G * dk * in_b + H * dv * in_b + 2 * H * 4 + H * dv * in_b)


def bench_gdn(torch, m, args):
    """Gated delta rule layer: in-place decode (tok/s, HBM roofline), the replay
    pool used for plain decode (verify of one token + commit, window W), and
    speculative verify + commit with T drafts, each in its own timed region."""
    c = GDN
    H, G, dk, dv, R, T = c["H"], c["G"], c["dk"], c["dv"], c["R"], c["tokens"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 171 + 17 * args.rank)
    stream = torch.cuda.current_stream()
    q, k, v, g, beta = gdn_inputs(torch, gen, T * R, H, G, dk, dv)
    q, k, v, g, beta = (t.view(T, R, *t.shape[1:]) for t in (q, k, v, g, beta))
    y = torch.empty((R, H, dv), dtype=torch.bfloat16, device="cuda")
    slots = list(range(R))
    zeros = torch.zeros(R, dtype=torch.int32, device="cuda")
    out = {}

    def new_pool(W, T1, n):
        init = (torch.randn((n, H, dv, dk), generator=gen, device="cuda") * 0.1).contiguous()
        p = m.ssm_gdn_init(m.make_gdn_config(H, G, dk, dv, m.SSM_DTYPE_BF16, W, T1), n, init)
        del init
        return p

    def timed(fn, n):
        fn(min(n, 8))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(n)
        e1.record(stream)
        torch.cuda.synchronize()
        return 1000.0 * e0.elapsed_time(e1) / n

    # in place
    pool = new_pool(c["W"], 1, R)

    def decode(n):
        for t in range(n):
            assert m.ssm_gdn_decode_step(pool, slots, q[t % T], k[t % T], v[t % T], g[t % T], beta[t % T], y,
                                         stream=stream) == m.SSM_OK
    us = timed(decode, T)
    alg = algorithmic_bytes_gdn_decode(R, H, G, dk, dv)
    hbm_peak, _, peak_kind = measured_peaks()
    out["decode"] = dict(us_per_step=us, tok_per_s=R / (us / 1e6), achieved_gbs=alg / (us / 1e6) / 1e9,
                         algorithmic_bytes=alg, frac_of_hbm=alg / (us / 1e6) / 1e9 / hbm_peak,
                         hbm_peak_source=peak_kind)
    assert m.ssm_gdn_status(pool)[1] == 0
    m.ssm_gdn_destroy(pool)

    # replay pool used for plain decode
    pool = new_pool(c["W"], 1, R)
    yr = torch.empty((R, 1, H, dv), dtype=torch.bfloat16, device="cuda")

    def replay(n):
        for t in range(n):
            i = t % T
            assert m.ssm_gdn_verify_replay(pool, slots, 1, q[i], k[i], v[i], g[i], beta[i], yr,
                                           stream=stream) == m.SSM_OK
            assert m.ssm_gdn_commit(pool, slots, zeros, stream=stream) == m.SSM_OK
    out["replay_plain_decode_us_per_step"] = timed(replay, T)
    out["replay_speedup_over_decode"] = out["decode"]["us_per_step"] / out["replay_plain_decode_us_per_step"]
    assert m.ssm_gdn_status(pool)[1] == 0
    m.ssm_gdn_destroy(pool)
    del q, k, v, g, beta

    # speculative verify + commit, T drafts
    T1, S = c["T"] + 1, c["steps"]
    pool = new_pool(c["W"], T1, R)
    qs, ks, vs, gs, bs = gdn_inputs(torch, gen, 4 * R, H, G, dk, dv, n_tok=T1)
    qs, ks, vs, gs, bs = (t.view(4, R, *t.shape[1:]) for t in (qs, ks, vs, gs, bs))
    hits = torch.rand((S, R, c["T"]), generator=gen, device="cuda") < c["p"]
    acc = torch.where(hits.all(dim=2), torch.full((S, R), c["T"], device="cuda"),
                      (~hits).int().argmax(dim=2)).int().contiguous()
    yv = torch.empty((R, T1, H, dv), dtype=torch.bfloat16, device="cuda")

    def verify(n):
        for t in range(n):
            i = t % 4
            assert m.ssm_gdn_verify_replay(pool, slots, T1, qs[i], ks[i], vs[i], gs[i], bs[i], yv,
                                           stream=stream) == m.SSM_OK
            assert m.ssm_gdn_commit(pool, slots, acc[t % S], stream=stream) == m.SSM_OK
    out["replay_verify_us_per_step"] = timed(verify, S)
    out["replay_verify_over_decode"] = out["replay_verify_us_per_step"] / out["decode"]["us_per_step"]
    assert m.ssm_gdn_status(pool)[1] == 0
    m.ssm_gdn_destroy(pool)
    out["config"] = dict(batch=R, value_heads=H, key_heads=G, dk=dk, dv=dv, W=c["W"], T=c["T"], p=c["p"],
                         decode_tokens=T, verify_steps=S, dtype="bf16 q/k/v, fp32 g/beta/state")
    return out


def bench_graph_small_batch(torch, m, args, batches=(1, 8, 64), steps=32):
    """Launch cost at small batch: the same decode steps (and replay verify +
    commit steps) issued call by call from Python, and captured once as a
    CUDA graph of `steps` steps and replayed.  Device time per step with CUDA
    events around the whole loop, so host issue gaps count; capture_ms is the
    host time to capture and instantiate the graph."""
    c = DEC
    H, P, N, G = c["H"], c["P"], c["N"], c["G"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED + 151 + 17 * args.rank)
    A, D = head_params(torch, gen, H)
    stream = torch.cuda.current_stream()
    out = {}

    def timed(fn, reps=3):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return 1000.0 * best / steps

    def measure(pool, body):
        body(pool)  # first calls outside the capture
        torch.cuda.synchronize()
        eager_us = timed(lambda: body(pool))
        g = torch.cuda.CUDAGraph()
        t0 = time.perf_counter()
        with torch.cuda.graph(g):
            body(pool)
        torch.cuda.synchronize()
        capture_ms = 1000.0 * (time.perf_counter() - t0)
        g.replay()
        graph_us = timed(g.replay)
        st, flags = m.ssm_pool_status(pool)
        assert st == m.SSM_OK and flags == 0, f"graph bench raised device flags {flags}"
        return dict(eager_us_per_step=eager_us, graph_us_per_step=graph_us, capture_ms=capture_ms,
                    graph_speedup=eager_us / graph_us)

    for R in batches:
        slots = list(range(R))
        x, dt, B, C = step_inputs(torch, gen, steps * R, H, P, G, N)
        x, dt, B, C = (t.view(steps, R, *t.shape[1:]) for t in (x, dt, B, C))
        y = torch.empty((steps, R, H, P), dtype=torch.bfloat16, device="cuda")
        pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_F32, m.SSM_MODE_COPY, 16, 1),
                                R)

        def decode(p):
            for s in range(steps):
                assert m.ssm_decode_step(p, slots, x[s], dt[s], B[s], C[s], A, D, y[s]) == m.SSM_OK

        out[f"decode_b{R}"] = measure(pool, decode)
        m.ssm_state_destroy(pool)
        del x, dt, B, C, y

    R, T1, W = 8, 9, 16
    slots = list(range(R))
    x, dt, B, C = step_inputs(torch, gen, steps * R, H, P, G, N, n_tok=T1)
    x, dt, B, C = (t.view(steps, R, *t.shape[1:]) for t in (x, dt, B, C))
    y = torch.empty((steps, R, T1, H, P), dtype=torch.bfloat16, device="cuda")
    acc = torch.randint(0, T1, (steps, R), generator=gen, device="cuda", dtype=torch.int32)
    pool = m.ssm_state_init(m.make_config(H, P, N, G, m.SSM_DTYPE_BF16, m.SSM_DTYPE_F32, m.SSM_MODE_REPLAY, W, T1), R)

    def verify(p):
        for s in range(steps):
            assert m.ssm_verify_replay(p, slots, T1, x[s], dt[s], B[s], C[s], A, D, y[s]) == m.SSM_OK
            assert m.ssm_state_commit(p, slots, acc[s], False, A) == m.SSM_OK

    out[f"replay_verify_commit_b{R}_T{T1 - 1}"] = measure(pool, verify)
    m.ssm_state_destroy(pool)
    out["config"] = dict(heads=H, headdim=P, dstate=N, groups=G, steps_per_graph=steps, verify_W=W,
                         timing="best of 3 loops, CUDA events around the loop")
    return out


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: implementer and part codes)."""
    try:
        text = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    m = re.search(r"^model name\s*:\s*(.+)$", text, flags=re.M)
    if m:
        return m.group(1).strip()
    imp = re.search(r"^CPU implementer\s*:\s*(\S+)", text, flags=re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", text, flags=re.M)
    if imp and part:
        return f"Arm implementer {imp.group(1)} part {part.group(1)}"
    return "unknown"


def _cpu_inputs(R, T1, H, P, N, G, seed):
    """Widened (exact) bf16 x / B / C and fp32 dt of R requests x T1 tokens, from synth."""
    import synth
    x, dt, B, C = synth.batch_tokens(seed, 0, R, T1, H, P, G, N, synth.BF16, synth.F32)
    return (synth.widen(x, synth.BF16), synth.widen(dt, synth.F32), synth.widen(B, synth.BF16),
            synth.widen(C, synth.BF16))


def _time_cpu(fn, budget_s):
    """Run fn() (one unit of work, returning the units it did) until about budget_s has passed."""
    units, t0 = 0, time.perf_counter()
    while True:
        units += fn()
        el = time.perf_counter() - t0
        if el >= budget_s:
            return units, el


def cpu_workloads(budget_s=1.5):
    """The oracle's fp32 instantiation (the same loops with fp32 values and
    accumulators, OpenMP over independent (request, head) pairs, or a thread
    per (sequence, head) for the scans) on the host cores, on bounded samples
    of each workload, on all cores and on one core.  Rates are scaled to each
    workload's own unit (tokens per second, or microseconds per step of the
    whole batch)."""
    import concurrent.futures as cf

    import numpy as np

    import oracle
    import synth
    all_cores = oracle.f32_threads()
    out = {}
    # decode (batch 256 at Nemotron heads): tok/s
    c = DEC
    H, P, N, G = c["H"], c["P"], c["N"], c["G"]
    A, D = synth.head_params(SEED, H)
    x, dt, B, C = (a[:, 0] for a in _cpu_inputs(32, 1, H, P, N, G, SEED + 1))
    for name, n_thr in (("all_cores", all_cores), ("one_core", 1)):
        oracle.f32_set_threads(n_thr)
        R = 32 if n_thr > 1 else 4
        st = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(R)]).astype(np.float32)
        xs, dts, Bs, Cs = x[:R], dt[:R], B[:R], C[:R]
        units, el = _time_cpu(lambda: (oracle.f32_decode_step(st, xs, dts, Bs, Cs, A, D), R)[1], budget_s)
        out.setdefault("decode", {})[name] = dict(value=units / el, unit="tok/s", threads=n_thr,
                                                   sample=f"{R} requests x all {H} heads per token")
    # speculative verify at batch 512, T = 8 (copy: T+1 states written; replay: checkpoint + log, fold when
    # the window fills): microseconds per verify step of all 512 requests
    v = VER
    T1, W, Rfull = v["T"] + 1, v["W"], v["R"]
    xs, dts, Bs, Cs = _cpu_inputs(8, T1, H, P, N, G, SEED + 2)
    acc = synth.accept_counts(SEED, 64, 8, v["T"], v["p"])
    Wc = W - 1 + T1
    for name, n_thr in (("all_cores", all_cores), ("one_core", 1)):
        oracle.f32_set_threads(n_thr)
        R = 8 if n_thr > 1 else 1
        st = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(R)]).astype(np.float32)
        units, el = _time_cpu(lambda: (oracle.f32_verify_copy(st, xs[:R], dts[:R], Bs[:R], Cs[:R], A, D), R)[1],
                              budget_s)
        out.setdefault("verify_copy_b512", {})[name] = dict(
            value=1e6 * el / units * Rfull, unit="us/step", threads=n_thr,
            sample=f"{R} requests x 1 verify step of {T1} tokens (T={v['T']}), scaled to {Rfull} requests")
        lx = np.zeros((R, Wc, H, P), np.float32)
        ldt = np.zeros((R, Wc, H), np.float32)
        lB = np.zeros((R, Wc, G, N), np.float32)
        k = np.zeros(R, np.int32)
        step = [0]

        def replay_step():  # verify, then the commit rule: append below the window, else fold
            s_ = step[0] % 64
            oracle.f32_verify_replay(st, k, lx, ldt, lB, xs[:R], dts[:R], Bs[:R], Cs[:R], A, D)
            cnt = acc[s_][:R] + 1
            fold = (k + cnt >= W).astype(np.int32)
            if fold.any():
                oracle.f32_fold(st, k, cnt, fold, lx, ldt, lB, xs[:R], dts[:R], Bs[:R], A)
            for r in range(R):
                if fold[r]:
                    k[r] = 0
                else:
                    lx[r, k[r]:k[r] + cnt[r]] = xs[r, :cnt[r]]
                    ldt[r, k[r]:k[r] + cnt[r]] = dts[r, :cnt[r]]
                    lB[r, k[r]:k[r] + cnt[r]] = Bs[r, :cnt[r]]
                    k[r] += cnt[r]
            step[0] += 1
            return R
        units, el = _time_cpu(replay_step, budget_s)
        out.setdefault("verify_replay_b512", {})[name] = dict(
            value=1e6 * el / units * Rfull, unit="us/step", threads=n_thr,
            sample=f"{R} requests x {step[0]} verify + commit steps (T={v['T']}, p={v['p']}, W={W}), "
                   f"scaled to {Rfull} requests")
    # prefill: one thread per (sequence, head) sequential scan; tok/s of the whole layer
    for key, (Hh, L) in (("prefill_130m", (PRE["H"], 512)), ("prefill_2p7b_varlen", (80, 512))):
        xs, dts, Bs, Cs = (np.ascontiguousarray(a[0], np.float32) for a in _cpu_inputs(1, L, Hh, 64, 128, 1, SEED + 3))
        Ah, Dh = synth.head_params(SEED, Hh)
        for name, n_thr in (("all_cores", all_cores), ("one_core", 1)):
            heads = list(range(Hh)) if n_thr > 1 else [0, 1]

            def scan_all():
                y = np.empty((L, Hh, 64), np.float32)

                def one(h):
                    st = np.zeros((64, 128), np.float32)
                    oracle.f32_scan_head(st, xs[:, h], dts[:, h], Bs[:, 0], Cs[:, 0], Ah[h], Dh[h],
                                         Hh * 64, Hh, 128, y[:, h], Hh * 64)
                with cf.ThreadPoolExecutor(max_workers=n_thr) as ex:
                    list(ex.map(one, heads))
                return L * len(heads) / Hh  # tokens of the whole layer (all heads)
            units, el = _time_cpu(scan_all, budget_s)
            out.setdefault(key, {})[name] = dict(value=units / el, unit="tok/s", threads=n_thr,
                                                 sample=f"1 sequence x {L} tokens x {len(heads)} of {Hh} heads")
    oracle.f32_set_threads(all_cores)
    return out


def cpu_baseline(budget_s=1.5):
    """CPU baseline of every workload (the oracle's fp32 instantiation on all
    host cores and on one), with the decode rate on all cores as the headline."""
    w = cpu_workloads(budget_s)
    dec = w["decode"]["all_cores"]
    return dict(value=dec["value"], unit="tok/s", cores=dec["threads"], cpu=cpu_model(), kind="oracle",
                precision="fp32 values and accumulators (the fp64 parity oracle is not the speed baseline)",
                sample=dec["sample"], workloads=w)


# ---------------------------------------------------------------------------

def run_case(args):
    """One workload alone, small enough for a profiler capture: a few
    iterations, one short text line (no benchmark JSON)."""
    import torch

    import hybrid_serving_mamba_gb300 as m
    torch.cuda.set_device(0)
    args.rank = 0
    if args.case == "decode":
        DEC["R"] = args.batch or DEC["R"]
        DEC["tokens"] = 4
        args.steps, args.warmup = 1, 1
        out = bench_decode(torch, m, None, args, ClockSampler(0))
        print(json.dumps({"case": "decode", "batch": DEC["R"], "launch_us": 1000 * out["launch_ms"],
                          "bytes_per_launch": out["bytes_per_launch"]}))
    elif args.case == "verify":
        VER["R"] = args.batch or VER["R"]
        VER["steps"] = 4
        out = bench_verify(torch, m, args, T=args.T or None, windows=[args.W] if args.W else None)
        print(json.dumps({"case": "verify", "batch": VER["R"], "copy_us": out["copy"]["us_per_step"],
                          "replay_us": {w: r["us_per_step"] for w, r in out["replay"].items()},
                          "fold_in_verify_us": {w: r["us_per_step"] for w, r in out["replay_fold_in_verify"].items()}}))
    elif args.case == "prefill":
        PRE["R"] = args.batch or PRE["R"]
        out = bench_prefill(torch, m, args)
        print(json.dumps({"case": "prefill", "seqs": PRE["R"], "us": out["us_per_scan"], "path": out["path"]}))
    elif args.case == "prefill_varlen":
        out = bench_prefill_varlen(torch, m, args, chunk=args.chunk or 1024, S=args.batch or 64)
        print(json.dumps({"case": "prefill_varlen", "ms": out["ms_per_wave"], "path": out["path"]}))
    elif args.case == "graph":
        print(json.dumps({"case": "graph", **bench_graph_small_batch(torch, m, args)}))
    elif args.case == "gdn":
        GDN["R"] = args.batch or GDN["R"]
        print(json.dumps({"case": "gdn", **bench_gdn(torch, m, args)}))
    else:
        raise SystemExit(f"unknown case {args.case}")
    return 0


def run_reference(args):
    """The oracle as the reference arm: rank 0 times its fp32 instantiation
    (OpenMP over (request, head) on all host cores) on the decode workload,
    W untimed warm-up steps and K timed steps, each step a bounded sample of
    the batch-256 decode (a few requests, all heads, one token)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import synth
    steps, warmup = max(1, args.steps), max(0, args.warmup)
    c = DEC
    H, P, N, G = c["H"], c["P"], c["N"], c["G"]
    A, D = synth.head_params(SEED, H)
    R = 16
    st = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(R)]).astype(np.float32)
    x, dt, B, C = (a[:, 0] for a in _cpu_inputs(R, 1, H, P, N, G, SEED + 1))
    cores = oracle.f32_threads()

    def one_step():
        t0 = time.perf_counter()
        oracle.f32_decode_step(st, x, dt, B, C, A, D)
        return time.perf_counter() - t0

    for _ in range(warmup):
        one_step()
    secs = [one_step() for _ in range(steps)]
    total = sum(secs)
    v = R * steps / total
    sample = f"{R} of the 256 requests x all {H} heads, one decode token per step (fp32 oracle, OpenMP)"
    line = {"impl": "reference", "metric": "decode state-update tok/s", "value": v, "unit": "tok/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": warmup, "ms_per_step": 1000 * total / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "batched decode, 256 requests x 64 successive tokens, heads 128 x headdim 64 x "
                                   "dstate 128, 8 groups, bf16 x/B/C, fp32 dt and state (sampled requests)",
                       "l2": "state > L2"},
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def job_rate(local_ms, local_units, dist=None, device="cpu"):
    """Whole-job rate of N replicas: the units all ranks processed divided by
    the slowest rank's time (max over ranks); returns (rate per second, ms)."""
    ms, world = float(local_ms), 1
    if dist is not None:
        import torch
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, world = float(t.item()), dist.get_world_size()
    return local_units * world / (ms / 1000.0), ms


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-extras", action="store_true", help="decode only (no verify / prefill / e2e / cpu)")
    ap.add_argument("--case", choices=("decode", "verify", "prefill", "prefill_varlen", "graph", "gdn"),
                    help="run one workload alone (for profiler captures)")
    ap.add_argument("--batch", type=int, default=0, help="batch / sequence count of --case")
    ap.add_argument("--T", type=int, default=0, help="drafts per verify step of --case verify")
    ap.add_argument("--chunk", type=int, default=0, help="user chunk of --case prefill_varlen (256 or 1024)")
    ap.add_argument("--W", type=int, default=0, help="replay window of --case verify")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    if args.warmup < 3:
        args.warmup = 3

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    args.rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    import hybrid_serving_mamba_gb300 as m  # fails loudly without the built library

    clocks = ClockSampler(local)
    dec = bench_decode(torch, m, dist, args, clocks)
    value, ms = job_rate(dec["ms"], dec["tokens"], dist, "cuda")
    hbm_peak, _, peak_kind = measured_peaks()
    achieved = dec["bytes_per_launch"] / (dec["launch_ms"] / 1000.0) / 1e9
    traffic = profiled_traffic("decode_kernel_nemotron_b256.md", "hybrid_serving_mamba_gb300/csrc/step_kernels.cu",
                               "hybrid_serving_mamba_gb300/csrc/ssm_internal.cuh")

    extras = {}
    if not args.no_extras:
        extras["verify_b512"] = bench_verify(torch, m, args, static=True)
        extras["verify_b512_sweep"] = bench_verify_sweep(torch, m, args)
        extras["prefill"] = bench_prefill(torch, m, args)
        extras["prefill_varlen"] = bench_prefill_varlen(torch, m, args, chunk=1024)
        extras["prefill_varlen_chunk256"] = bench_prefill_varlen(torch, m, args, chunk=256)
        extras["replay_plain_decode_b256"] = bench_replay_plain_decode(torch, m, args)
        extras["graph_small_batch"] = bench_graph_small_batch(torch, m, args)
        extras["gdn_b256"] = bench_gdn(torch, m, args)
        e2e = bench_decode_e2e(torch, m, args)
    else:
        e2e = None
    if args.rank != 0:
        if dist is not None:
            dist.barrier()
        return 0
    line = {
        "metric": "decode state-update tok/s",
        "value": value,
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded, drawn on device)",
        "config": {"workload": "batched decode, 256 requests x 64 successive tokens, heads 128 x headdim 64 x "
                               "dstate 128, 8 groups, bf16 x/B/C, fp32 dt and state",
                   "batch": DEC["R"], "tokens_per_step": DEC["R"] * DEC["tokens"], "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (1 GiB state per replica)"},
        "hbm_gbs": dec["bytes_per_launch"] * dec["launches"] / (dec["ms"] / 1000.0) / 1e9,
        "roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "peak_source": peak_kind,
                     "traffic": traffic, "algorithmic_bytes_per_launch": dec["bytes_per_launch"],
                     "launch_us": 1000 * dec["launch_ms"]},
        "clocks": dec["clocks"],
        "gpu_launches": dec["launches"],
    }
    if e2e is not None:
        line["e2e"] = {"value": e2e["tokens"] / (e2e["ms"] / 1000.0), "unit": "tok/s",
                       "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "entry": "ssm_decode_steps_host", "steps": args.steps}
    line.update(extras)
    if not args.no_extras:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
    return 0


if __name__ == "__main__":
    sys.exit(main())
