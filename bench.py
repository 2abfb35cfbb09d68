#!/usr/bin/env python
"""Benchmark of the Gated DeltaNet mixer hot path on one GB300 (or N replicas).

A step is one pass of the whole prefill path on the prefill workload
(B=1, T=4096, Nk=16 -> Nv=32, Dk=Dv=128, C=8192, bf16, fp32 gates/state):
gdn_conv_gating (+ conv-state output) -> gdn_chunk_prefill -> gdn_gated_rmsnorm.
The single call gdn_chunk_prefill_gated_norm (chunk prefill with the norm in its
epilogue) is timed beside it.
The fused decode step (B=256, one token each, fp32 state in place) is timed in
the same run and reported under "decode" (median of per-step events, with the
spread), and the same prefill path on the packed workload (16 sequences,
lengths ~ U[512, 8192]) and on the long one (T=131072) under "varlen" and
"long_context" (tokens/s, the chunk call's TFLOP/s and fraction of peak, and
the oracle's tokens/s on a bounded sample).  Every device time is the median of
--steps timed replays.  "e2e" is the same prefill step through
the public API with the inputs copied in from pinned host memory and y read back
every step; the copies of step i+1 run on one copy stream under step i's compute
and the read-backs on a second (two device buffer sets), as a pipelined caller would
run them.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-cpu-baseline] [--headline-only]

--impl reference times the fp64 CPU oracle (the reference arm of this
project) on a bounded sample of the same workload.  Under torchrun (N > 1)
every rank runs its own replica (the path has no exchange step); rank 0
prints one JSON line.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = 'GDN prefill tokens/s & % bf16 TC peak; decode tokens/s & HBM GB/s vs ~8TB/s'
CHUNK = 64
L2_FLUSH_BYTES = 512 << 20
NOMINAL_HBM_GBS = 8000.0


def chunk_flops_per_chunk_head(Dk, Dv, C=CHUNK):
    """Algorithmic flops of one chunk of one value head: KK^T, QK^T, W, U~ and
    P.U over full 64x64 tiles, W.S, Q.S and K^T.U, and the triangular inverse."""
    return 2 * C * C * (3 * Dk + 2 * Dv) + 6 * C * Dk * Dv + C ** 3 / 3.0


def chunk_flops(lengths, Nv, Dk, Dv):
    return sum(math.ceil(L / CHUNK) for L in lengths) * Nv * chunk_flops_per_chunk_head(Dk, Dv)


def chunk_bytes(tokens, Nk, Nv, Dk, Dv, act=2, out=2):
    # q, k read once per key head, v once, g and beta fp32, o written once
    return tokens * (2 * Nk * Dk * act + Nv * Dv * act + 2 * Nv * 4 + Nv * Dv * out)


def rmsnorm_bytes(rows, dim, act=2, out=2):
    return rows * dim * (act + act + out) + dim * 4


def code_hash(src):
    """sha1 of a C++/CUDA source with comments and whitespace removed: a counter capture stays
    attached to its kernel through edits of the comments only."""
    import hashlib
    import re
    src = re.sub(r'/\*.*?\*/', ' ', src, flags=re.S)
    src = re.sub(r'//[^\n]*', ' ', src)
    return hashlib.sha1(' '.join(src.split()).encode()).hexdigest()


def conv_gating_bytes(tokens, num_seqs, C, Nk, Nv, Dk, Dv, act=2):
    return (tokens * (C * act + 2 * Nv * act)            # mixed_qkv, a, b
            + tokens * (2 * Nk * Dk + Nv * Dv) * act      # q, k, v out
            + tokens * Nv * 2 * 4                         # g, beta out
            + C * 4 * act + num_seqs * C * 3 * act)       # weights, conv state out


def decode_bytes(B, Nk, Nv, Dk, Dv, act=2, out=2):
    C = 2 * Nk * Dk + Nv * Dv
    return (2 * B * Nv * Dk * Dv * 4            # state read + write
            + 2 * B * C * 3 * act               # conv state read + write
            + B * C * act                       # mixed_qkv
            + B * Nv * Dv * act                 # z
            + 2 * B * Nv * act                  # a, b
            + B * Nv * Dv * out                 # y
            + C * 4 * act + 2 * Nv * 4 + Dv * 4)  # weights


def load_peaks():
    p = os.path.join(ROOT, 'MEASURED_PEAKS.json')
    if os.path.exists(p):
        d = json.load(open(p))
        return d['hbm_gbs'], d['bf16_tflops'], d.get('bf16_tflops_sustained', d['bf16_tflops']), 'measured'
    return 6800.0, 1900.0, 1700.0, 'fallback'


class ClockSampler:
    FIELDS = ('index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,'
              'clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,'
              'clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu')

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix='.csv')
            os.close(fd)
            self.proc = subprocess.Popen(
                ['nvidia-smi', '-i', str(self.gpu), '--query-gpu=' + self.FIELDS,
                 '--format=csv,noheader,nounits', '-lms', '100'],
                stdout=open(self.path, 'w'), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {'sm_mhz': None, 'sm_max_mhz': None, 'reasons': ['nvidia-smi unavailable']}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return summarize_clocks(lines)


def summarize_clocks(lines):
    """The clock record of a run from nvidia-smi's csv rows (ClockSampler.FIELDS, no header or
    units): the median SM clock over the samples under load (the GPU busy for at least half of
    the sample period by its utilization counter; all samples if none is), the maximum clock,
    and every throttle reason seen active."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(',')]
        if len(parts) < 9:
            continue
        try:
            row = (float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9])
        except ValueError:
            continue
        try:
            util = float(parts[9]) if len(parts) > 9 else None
        except ValueError:
            util = None
        rows.append(row + (util,))
    if not rows:
        return {'sm_mhz': None, 'sm_max_mhz': None, 'reasons': [], 'samples': 0}
    names = ['hw_slowdown', 'hw_thermal_slowdown', 'sw_thermal_slowdown', 'sw_power_cap']
    reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == 'active'})
    loaded = [r for r in rows if r[4] is not None and r[4] >= 50.0] or rows
    return {'sm_mhz': statistics.median(r[0] for r in loaded), 'sm_max_mhz': max(r[1] for r in rows),
            'reasons': reasons, 'samples': len(rows), 'samples_under_load': len(loaded),
            'power_w_max': max(r[2] for r in rows)}


def dist_setup():
    ws = int(os.environ.get('WORLD_SIZE', '1'))
    rank = int(os.environ.get('RANK', '0'))
    local = int(os.environ.get('LOCAL_RANK', '0'))
    return ws, rank, local


def make_ranks(dist, device):
    """barrier() and max_over_ranks(x) of the bench's replicas: `dist` is torch.distributed with
    an initialised process group (NCCL on GPUs, gloo in the CPU tests) or None for one process;
    `device` holds the reduction tensor and, when it is a GPU, is synchronised by barrier()."""
    import torch

    def barrier():
        if dist is not None:
            dist.barrier()
        if device.type == 'cuda':
            torch.cuda.synchronize(device)

    def max_over_ranks(x):
        if dist is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_over_ranks


def whole_job_rate(units_per_rank, world_size, ms_max):
    """Units processed by all ranks per second, over the slowest rank's time (weak scaling)."""
    return units_per_rank * world_size / (ms_max * 1e-3)


# ------------------------------------------------------------------ reference arm

def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_prefill_sample(inp, ntok):
    """The oracle's prefill over the first ntok tokens of the workload's first sequence (all
    heads, from that sequence's initial recurrent state)."""
    import numpy as np
    import oracle as O
    sh = inp.shape
    ntok = min(ntok, inp.lengths[0])
    f = lambda t: t[:ntok].to(dtype=__import__('torch').float64).numpy()  # noqa: E731
    g = lambda t: t.to(dtype=__import__('torch').float64).numpy()  # noqa: E731
    S0 = None if inp.S0 is None else g(inp.S0[:1])
    r = O.mixer_prefill(f(inp.mixed_qkv), g(inp.conv_w), f(inp.a), f(inp.b), g(inp.A_log),
                        g(inp.dt_bias), f(inp.z), g(inp.norm_w), sh.Nk, sh.Nv, sh.Dk, sh.Dv,
                        initial_state=S0)
    return np.asarray(r['y']).shape[0]


def cpu_baseline(inp, budget_s=12.0, name='prefill_t4096'):
    """Oracle tokens/s on a bounded prefix of the workload's first sequence."""
    n = 32
    t0 = time.perf_counter()
    oracle_prefill_sample(inp, n)
    dt = time.perf_counter() - t0
    ntok = int(max(32, min(inp.lengths[0], n * budget_s / max(dt, 1e-3))))
    t0 = time.perf_counter()
    ntok = oracle_prefill_sample(inp, ntok)
    dt = time.perf_counter() - t0
    return {'value': ntok / dt, 'unit': 'tokens/s', 'cores': cpu_threads(), 'kind': 'oracle',
            'sample': 'fp64 NumPy oracle prefill (conv_gating + token-by-token recurrence + gated '
                      'RMSNorm) over the first %d tokens of %s (first sequence), all %d heads, %.1f s'
                      % (ntok, name, inp.shape.Nv, dt)}


def cpu_baseline_decode(dinp, budget_s=3.0):
    """Oracle tokens/s of the fused decode step (one token per sequence) on a bounded number
    of the workload's sequences."""
    import numpy as np
    import oracle as O
    sh = dinp.shape
    f64 = lambda t: t.detach().to('cpu').double().numpy()  # noqa: E731
    args = [f64(t) for t in (dinp.mixed_qkv, dinp.conv_w, dinp.conv_state, dinp.a, dinp.b, dinp.A_log,
                             dinp.dt_bias, dinp.S0, dinp.z, dinp.norm_w)]

    def run(n):
        sub = [x[:n] if i in (0, 2, 3, 4, 7, 8) else x for i, x in enumerate(args)]
        O.decode_step(*sub, sh.Nk, sh.Nv, sh.Dk, sh.Dv)

    n = 4
    t0 = time.perf_counter()
    run(n)
    dt = time.perf_counter() - t0
    n = int(max(1, min(dinp.num_seqs, n * budget_s / max(dt, 1e-3))))
    t0 = time.perf_counter()
    run(n)
    dt = time.perf_counter() - t0
    return {'value': n / dt, 'unit': 'tokens/s', 'cores': cpu_threads(), 'kind': 'oracle',
            'sample': 'fp64 NumPy oracle decode step (conv update, gates, recurrence, gated RMSNorm) '
                      'for %d of the %d sequences of decode_b256, %.1f s' % (n, dinp.num_seqs, dt)}


# Kernels of this library per call on the tensor-core path: conv_gating launches one (with no
# conv state in, its tiled pass writes the new state); chunk prefill launches one for a single
# sequence (the cooperative solve + scan launch) and two for a packed batch (solve, then scan);
# the gated norm one.
def chunk_launches(num_seqs):
    return 1 if num_seqs == 1 else 2


def time_prefill_workload(name, steps, warmup, barrier, max_over_ranks, tc_peak):
    """The prefill path (conv_gating -> chunk_prefill -> gated_rmsnorm) on a workload whose
    inputs exceed L2 (no flush needed between steps): median device time of the step and of
    the chunk call alone, each replayed from a CUDA graph with one event pair per replay."""
    import torch
    from gated_deltanet_linear_conv_gb300 import gdn
    from gated_deltanet_linear_conv_gb300 import inputs as I

    inp = I.workload(name)
    sh = inp.shape
    T, N = inp.total_tokens, inp.num_seqs
    bf = torch.bfloat16
    dev = lambda t: None if t is None else t.cuda()  # noqa: E731
    x, w, a, b = dev(inp.mixed_qkv), dev(inp.conv_w), dev(inp.a), dev(inp.b)
    A_log, dt_bias, z, nw = dev(inp.A_log), dev(inp.dt_bias), dev(inp.z), dev(inp.norm_w)
    cu = dev(inp.cu_seqlens()) if N > 1 else None
    S0 = dev(inp.S0)
    ST = torch.empty(N, sh.Nv, sh.Dk, sh.Dv, device='cuda')
    cs_out = torch.empty(N, sh.C, 3, dtype=bf, device='cuda')
    bufs = dict(q=torch.empty(T, sh.Nk, sh.Dk, dtype=bf, device='cuda'),
                k=torch.empty(T, sh.Nk, sh.Dk, dtype=bf, device='cuda'),
                v=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'),
                g=torch.empty(T, sh.Nv, device='cuda'), beta=torch.empty(T, sh.Nv, device='cuda'),
                o=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'),
                y=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'))
    ws_bytes = gdn.chunk_prefill_workspace_size(N, T, sh.Nk, sh.Nv, sh.Dk, sh.Dv)
    wsp = torch.empty(ws_bytes, dtype=torch.uint8, device='cuda') if ws_bytes else None

    def chunk_call():
        gdn.chunk_prefill(bufs['q'], bufs['k'], bufs['v'], bufs['g'], bufs['beta'], 1.0, S0, ST, cu, N,
                          bf, bufs['o'], wsp)

    def step():
        gdn.conv_gating(x, w, a, b, A_log, dt_bias, sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=cu, num_seqs=N,
                        conv_state_out=cs_out, out=(bufs['q'], bufs['k'], bufs['v'], bufs['g'], bufs['beta']))
        chunk_call()
        gdn.gated_rmsnorm(bufs['o'], z, nw, 1e-6, bf, bufs['y'])

    for _ in range(warmup):
        step()
    barrier()
    graphs = {}
    for key, fn in (('step', step), ('chunk', chunk_call)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[key] = g
    stream = torch.cuda.current_stream()
    res = {}
    for key, g in graphs.items():
        g.replay()
        barrier()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in evs:
            e0.record(stream)
            g.replay()
            e1.record(stream)
        barrier()
        res[key] = max_over_ranks(statistics.median(e0.elapsed_time(e1) for e0, e1 in evs))
    gdn.check_device_error()
    flops = chunk_flops(inp.lengths, sh.Nv, sh.Dk, sh.Dv)
    tflops = flops / (res['chunk'] * 1e-3) / 1e12
    launches = (steps + warmup) * (2 + chunk_launches(N)) + steps * chunk_launches(N)
    out = {'workload': name, 'num_seqs': N, 'tokens': T,
           'lengths': inp.lengths if N > 1 else None,
           'tokens_per_s': whole_job_rate(T, 1, res['step']),
           'us_per_step': res['step'] * 1e3, 'us_chunk_prefill': res['chunk'] * 1e3,
           'chunk_prefill': {'TFLOP/s': tflops, 'frac_tc': tflops / tc_peak,
                             'algorithmic_flops': flops,
                             'flops_formula': 'per sequence ceil(L/64) chunks x Nv x '
                                              '(2*64^2*(3Dk+2Dv) + 6*64*Dk*Dv + 64^3/3)'},
           'workspace_bytes': ws_bytes,
           'timing': 'cuda-graph replay, median of %d, inputs larger than L2 (no flush)' % steps}
    del graphs, bufs, wsp, x, z
    torch.cuda.empty_cache()
    return out, inp, launches


def run_reference(args):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    from gated_deltanet_linear_conv_gb300 import inputs as I
    inp = I.workload('prefill_t4096')
    ntok = 64
    for _ in range(args.warmup):
        oracle_prefill_sample(inp, ntok)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_prefill_sample(inp, ntok)
    dt = (time.perf_counter() - t0) / args.steps
    value = ntok / dt
    line = {'impl': 'reference', 'metric': METRIC, 'value': value, 'unit': 'tokens/s',
            'n_gpus': ws, 'steps': args.steps, 'warmup': args.warmup, 'ms_per_step': dt * 1e3,
            'higher_is_better': True, 'scaling': 'weak', 'vs_baseline': None, 'dtype': 'f64',
            'data': 'synthetic',
            'config': {'workload': 'prefill_t4096', 'B': 1, 'T': 4096, 'Nk': 16, 'Nv': 32, 'Dk': 128,
                       'Dv': 128, 'chunk': CHUNK, 'sample_tokens_per_step': ntok},
            'cpu_baseline': {'value': value, 'unit': 'tokens/s', 'cores': cpu_threads(), 'kind': 'oracle',
                             'sample': 'first %d tokens of the prefill workload per step' % ntok},
            'e2e': {'value': value, 'unit': 'tokens/s', 'h2d_bytes_per_step': 0, 'd2h_bytes_per_step': 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import torch
    from gated_deltanet_linear_conv_gb300 import gdn
    from gated_deltanet_linear_conv_gb300 import inputs as I

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group('nccl', device_id=torch.device('cuda', local))

    barrier, max_over_ranks = make_ranks(dist, torch.device('cuda', local))

    hbm_peak, tc_peak, tc_sust, peak_src = load_peaks()
    sampler = ClockSampler(local)

    # ---------------- prefill workload, resident in HBM
    inp = I.workload('prefill_t4096')
    sh = inp.shape
    T = inp.total_tokens
    dev = lambda t: t.cuda()  # noqa: E731
    x, w, a, b = dev(inp.mixed_qkv), dev(inp.conv_w), dev(inp.a), dev(inp.b)
    A_log, dt_bias, z, nw = dev(inp.A_log), dev(inp.dt_bias), dev(inp.z), dev(inp.norm_w)
    bf = torch.bfloat16
    bufs = dict(q=torch.empty(T, sh.Nk, sh.Dk, dtype=bf, device='cuda'),
                k=torch.empty(T, sh.Nk, sh.Dk, dtype=bf, device='cuda'),
                v=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'),
                g=torch.empty(T, sh.Nv, device='cuda'), beta=torch.empty(T, sh.Nv, device='cuda'),
                o=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'),
                y=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'))
    ws_bytes = gdn.chunk_prefill_workspace_size(1, T, sh.Nk, sh.Nv, sh.Dk, sh.Dv)
    if ws_bytes:
        bufs['workspace'] = torch.empty(ws_bytes, dtype=torch.uint8, device='cuda')
    conv_state_out = torch.empty(1, sh.C, 3, dtype=bf, device='cuda')
    final_state = torch.empty(1, sh.Nv, sh.Dk, sh.Dv, device='cuda')
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device='cuda')
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device='cuda')
    stream = torch.cuda.current_stream()

    def conv_call():
        gdn.conv_gating(x, w, a, b, A_log, dt_bias, sh.Nk, sh.Nv, sh.Dk, sh.Dv, num_seqs=1,
                        conv_state_out=conv_state_out,
                        out=(bufs['q'], bufs['k'], bufs['v'], bufs['g'], bufs['beta']))

    def chunk_call():
        gdn.chunk_prefill(bufs['q'], bufs['k'], bufs['v'], bufs['g'], bufs['beta'], 1.0, None, final_state,
                          None, 1, bf, bufs['o'], bufs.get('workspace'))

    def norm_call():
        gdn.gated_rmsnorm(bufs['o'], z, nw, 1e-6, bf, bufs['y'])

    def fused_call():          # chunk prefill with the gated RMSNorm in its epilogue (reported beside)
        gdn.chunk_prefill_gated_norm(bufs['q'], bufs['k'], bufs['v'], bufs['g'], bufs['beta'], z, nw, 1.0,
                                     None, final_state, None, 1, 1e-6, bf, bufs['y'], bufs.get('workspace'))

    def prefill_step():
        conv_call()
        chunk_call()
        norm_call()

    sampler.start()
    for _ in range(args.warmup):
        prefill_step()
    barrier()
    # Device time of the step and of each call: each is captured once in a CUDA
    # graph and replayed (the replay launches the same kernels on the same
    # buffers, without the host's per-call marshalling in between); the L2
    # flush runs before every timed replay.
    timing = 'cuda-graph replay'
    run = {'step': prefill_step, 'conv': conv_call, 'chunk': chunk_call, 'norm': norm_call, 'fused': fused_call}
    try:
        graphs = {}
        for name, fn in run.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            graphs[name] = g
        run = {name: g.replay for name, g in graphs.items()}
    except Exception as exc:  # capture refused: time the eager calls instead
        torch.cuda.synchronize()
        timing = 'eager calls (graph capture unavailable: %s)' % type(exc).__name__
    for fn in run.values():
        fn()
    barrier()
    stream = torch.cuda.current_stream()

    def timed(fn):
        evs = []
        for i in range(args.steps):
            # evict the inputs from L2 between steps: a 512 MiB write, then a 512 MiB read so that
            # the lines left in L2 are clean and the step does not pay for writing back the flush
            flush.fill_(float(i))
            flush_rd.sum()
            e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            e[0].record(stream)
            fn()
            e[1].record(stream)
            evs.append(e)
        barrier()
        return [e[0].elapsed_time(e[1]) for e in evs]

    t_step = timed(run['step'])
    t_conv = timed(run['conv'])
    t_chunk = timed(run['chunk'])
    t_norm = timed(run['norm'])
    t_fused = timed(run['fused'])
    ms_step = max_over_ranks(statistics.median(t_step))
    # Kernels of this library per call: conv_gating is one (the tiled pass writes the new conv
    # state itself when there is no state in, as here), chunk prefill one (one sequence: one
    # cooperative solve + scan launch), gated norm one, the fused chunk + norm call one.
    # Timed: the step replays, then the replays of each call and of the fused call.
    k_conv, k_chunk, k_norm, k_fused = 1, 1, 1, 1
    k_step = k_conv + k_chunk + k_norm
    launches_prefill = args.steps * (k_step + k_conv + k_chunk + k_norm + k_fused)

    # ---------------- decode workload (fused step, state in place; 512 MiB state > L2)
    del flush, flush_rd
    dinp = I.workload('decode_b256')
    B = dinp.num_seqs
    dx, dw, da, db = dev(dinp.mixed_qkv), dev(dinp.conv_w), dev(dinp.a), dev(dinp.b)
    dA, ddt, dz, dnw = dev(dinp.A_log), dev(dinp.dt_bias), dev(dinp.z), dev(dinp.norm_w)
    dcs, dS = dev(dinp.conv_state), dev(dinp.S0)
    dy = torch.empty(B, sh.Nv, sh.Dv, dtype=bf, device='cuda')

    def decode_step():
        gdn.decode_fused(dx, dw, dcs, da, db, dA, ddt, dS, dz, dnw, sh.Nk, sh.Nv, sh.Dk, sh.Dv,
                         out_dtype=bf, y=dy)

    dsteps = max(args.steps, 20)
    for _ in range(args.warmup):
        decode_step()
    barrier()
    # one event pair per step, the steps back to back (the 512 MiB state exceeds L2)
    dev_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(dsteps)]
    for e0_, e1_ in dev_evs:
        e0_.record(stream)
        decode_step()
        e1_.record(stream)
    barrier()
    t_dec = [a.elapsed_time(b) for a, b in dev_evs]
    ms_dec = max_over_ranks(statistics.median(t_dec))
    del dS, dcs

    # ---------------- end to end through the public API with host buffers
    pin = lambda t: t.pin_memory()  # noqa: E731
    hx, ha, hb, hz = pin(inp.mixed_qkv), pin(inp.a), pin(inp.b), pin(inp.z)
    hy = torch.empty(T, sh.Nv, sh.Dv, dtype=bf).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hx, ha, hb, hz))
    d2h = hy.numel() * hy.element_size()

    # Two sets of device inputs and outputs.  Step i's host->device copies run on one copy
    # stream while step i-1 computes, and step i's device->host read runs on a second one
    # after its compute, so that the two directions overlap.  (On a GB300 with a Grace host
    # the link moved about 208 GB/s host->device and 191 GB/s device->host, copy engines and
    # a copy kernel on mapped host memory alike; this step's traffic alone took 0.519 ms per
    # step with one upload stream beside the read-back, 0.528 ms with three.)  A copy into
    # set j waits for the compute that last read set j; a compute into set j waits for the
    # read-back of set j's previous result.  Every step still moves its own inputs and result
    # inside the timed region.
    sets = [(x, a, b, z, bufs['y'])]
    sets.append(tuple(torch.empty_like(t) for t in sets[0]))
    hys = [hy, torch.empty_like(hy).pin_memory()]
    h2d_stream = torch.cuda.Stream()
    d2h_stream = torch.cuda.Stream()
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    comp_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_h2d(j, first):
        with torch.cuda.stream(h2d_stream):
            if not first:
                h2d_stream.wait_event(comp_done[j])
            for dst, src in zip(sets[j][:4], (hx, ha, hb, hz)):
                dst.copy_(src, non_blocking=True)
            h2d_done[j].record(h2d_stream)

    def e2e_compute(j, first):
        xj, aj, bj, zj, yj = sets[j]
        stream.wait_event(h2d_done[j])
        if not first:
            stream.wait_event(d2h_done[j])
        gdn.conv_gating(xj, w, aj, bj, A_log, dt_bias, sh.Nk, sh.Nv, sh.Dk, sh.Dv, num_seqs=1,
                        conv_state_out=conv_state_out,
                        out=(bufs['q'], bufs['k'], bufs['v'], bufs['g'], bufs['beta']))
        chunk_call()
        gdn.gated_rmsnorm(bufs['o'], zj, nw, 1e-6, bf, yj)
        comp_done[j].record(stream)

    def e2e_d2h(j):
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(comp_done[j])
            hys[j].copy_(sets[j][4], non_blocking=True)
            d2h_done[j].record(d2h_stream)

    def e2e_steps(n, start=None):
        if start is not None:          # the first copies start inside the timed region
            h2d_stream.wait_event(start)
        e2e_h2d(0, True)
        for i in range(n):
            e2e_compute(i & 1, i < 2)
            if i + 1 < n:
                e2e_h2d((i + 1) & 1, i + 1 < 2)
            e2e_d2h(i & 1)
        stream.wait_event(d2h_done[(n - 1) & 1])     # (the read-backs run in order on one stream)

    e2e_steps(args.warmup)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(args.steps, e0)
    e1.record(stream)
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    # ---------------- the packed and the long-context prefill workloads (inputs > L2)
    del sets, hys
    torch.cuda.empty_cache()
    extra = {}
    extra_launches = 0
    for key, name in (() if args.headline_only else (('varlen', 'varlen_16seq'), ('long_context', 'prefill_t131072'))):
        res, winp, nl = time_prefill_workload(name, args.steps, args.warmup, barrier, max_over_ranks, tc_peak)
        res['tokens_per_s'] = whole_job_rate(res['tokens'], ws, res['us_per_step'] * 1e-3)
        extra[key] = (res, winp)
        extra_launches += nl
    clocks = sampler.stop()
    gdn.check_device_error()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    flops = chunk_flops(inp.lengths, sh.Nv, sh.Dk, sh.Dv)
    us_chunk = statistics.median(t_chunk) * 1e3
    us_conv = statistics.median(t_conv) * 1e3
    us_norm = statistics.median(t_norm) * 1e3
    us_fused = statistics.median(t_fused) * 1e3
    nb = rmsnorm_bytes(T * sh.Nv, sh.Dv)
    tflops = flops / (us_chunk * 1e-6) / 1e12
    cb = conv_gating_bytes(T, 1, sh.C, sh.Nk, sh.Nv, sh.Dk, sh.Dv)
    kb = chunk_bytes(T, sh.Nk, sh.Nv, sh.Dk, sh.Dv)
    dbytes = decode_bytes(B, sh.Nk, sh.Nv, sh.Dk, sh.Dv)
    dec_gbs = dbytes / (ms_dec * 1e-3) / 1e9
    traffic = None      # DRAM bytes per launch from an ncu capture of the same kernel code, else null
    tp = os.path.join(ROOT, 'profiles', 'traffic.json')
    if os.path.exists(tp):
        rec = json.load(open(tp)).get('chunk_prefill_t4096')
        if rec:
            src = ''.join(open(os.path.join(ROOT, f)).read() for f in rec['sources'])
            if code_hash(src) == rec['code_sha1']:
                traffic = rec['bytes_per_launch']
    line = {
        'metric': METRIC,
        'value': whole_job_rate(T, ws, ms_step),
        'unit': 'tokens/s',
        'n_gpus': ws, 'steps': args.steps, 'warmup': args.warmup,
        'ms_per_step': ms_step,
        'higher_is_better': True, 'scaling': 'weak', 'vs_baseline': None,
        'dtype': 'bf16', 'data': 'synthetic',
        'config': {'workload': 'prefill_t4096', 'B': 1, 'T': T, 'Nk': sh.Nk, 'Nv': sh.Nv, 'Dk': sh.Dk,
                   'Dv': sh.Dv, 'C': sh.C, 'chunk': CHUNK, 'state': 'fp32', 'gates': 'fp32',
                   'l2': 'flushed between timed steps (512 MiB write, then 512 MiB read: clean lines)', 'parallelism': 'replicas',
                   'timing': timing},
        'roofline': {'kernel': 'gdn_chunk_prefill (one cooperative solve + scan launch)', 'bound': 'tensor', 'achieved': tflops,
                     'peak': tc_peak, 'unit': 'TFLOP/s', 'frac': tflops / tc_peak,
                     'traffic': traffic, 'peak_source': peak_src + ' bf16 dense (burst)',
                     'algorithmic_flops_per_launch': flops, 'us_per_launch': us_chunk,
                     'hbm_gbs': kb / (us_chunk * 1e-6) / 1e9},
        'kernels': {
            'conv_gating': {'us': us_conv, 'GB/s': cb / (us_conv * 1e-6) / 1e9,
                            'frac_hbm': cb / (us_conv * 1e-6) / 1e9 / hbm_peak, 'bytes': cb},
            'chunk_prefill': {'us': us_chunk, 'TFLOP/s': tflops, 'frac_tc': tflops / tc_peak},
            'gated_rmsnorm': {'us': us_norm, 'GB/s': nb / (us_norm * 1e-6) / 1e9,
                              'frac_hbm': nb / (us_norm * 1e-6) / 1e9 / hbm_peak, 'bytes': nb},
            'chunk_prefill_gated_norm': {'us': us_fused, 'note': 'one call: chunk prefill and the gated norm (for one sequence the norm runs beside the scan)'}},
        'decode': {'workload': 'decode_b256', 'kernel': 'gdn_decode_fused', 'steps': dsteps,
                   'us_per_step': ms_dec * 1e3, 'tokens_per_s': whole_job_rate(B, ws, ms_dec),
                   'us_per_step_spread': {'min': min(t_dec) * 1e3, 'median': ms_dec * 1e3,
                                          'p90': sorted(t_dec)[int(0.9 * (len(t_dec) - 1))] * 1e3,
                                          'max': max(t_dec) * 1e3},
                   'roofline': {'bound': 'hbm', 'achieved': dec_gbs, 'peak': hbm_peak, 'unit': 'GB/s',
                                'frac': dec_gbs / hbm_peak, 'frac_of_8tbs': dec_gbs / NOMINAL_HBM_GBS,
                                'bytes_per_launch': dbytes}},
        'e2e': {'value': whole_job_rate(T, ws, ms_e2e), 'unit': 'tokens/s', 'h2d_bytes_per_step': h2d,
                'd2h_bytes_per_step': d2h, 'ms_per_step': ms_e2e},
        'gpu_launches': launches_prefill + dsteps + k_step * args.steps + extra_launches,
        'clocks': clocks,
    }
    for key, (res, winp) in extra.items():
        if ws == 1 and not args.no_cpu_baseline:
            res['cpu_baseline'] = cpu_baseline(winp, 5.0, res['workload'])
        line[key] = res
    if ws == 1 and not args.no_cpu_baseline:
        line['cpu_baseline'] = cpu_baseline(inp)
        line['decode']['cpu_baseline'] = cpu_baseline_decode(dinp)
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument('--gpus', type=int, default=1)
    ap.add_argument('--steps', type=int, default=20)
    ap.add_argument('--warmup', type=int, default=5)
    ap.add_argument('--impl', default='ours', choices=['ours', 'reference'])
    ap.add_argument('--no-cpu-baseline', action='store_true')
    ap.add_argument('--headline-only', action='store_true',
                    help='time only prefill_t4096 and decode_b256 (no varlen / long-context lines): '
                         'a small device footprint for profiler captures')
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == 'ours':
        print('note: warmup raised to 3', file=sys.stderr)
        args.warmup = 3
    if args.impl == 'reference':
        run_reference(args)
    else:
        from gated_deltanet_linear_conv_gb300 import _build
        _build.build()
        run_ours(args)


if __name__ == '__main__':
    main()
