"""Super-tile cluster runtime for the fp32 GEMM: scheduler, pods, job files.

This is the cluster path of the "@cluster" attribute page ("What runs today")
and of "Show HN: Phobos" ("The DAG Compiler", "The Cluster Prototype"). It is
rebuilt for one box that holds one GB300:
  - the planner and the pod executor are native (``phobos_cl_plan``,
    ``phobos_pod_run`` in libphobos_gemm.so, declared in
    include/phobos_cluster.h);
  - this module is the control plane around them;
  - the scheduler plans every output super-tile, deals the super-tiles round
    robin over the nodes, and publishes each node's segment (instruction
    list) in a TCPStore;
  - each pod is one process. It runs its segments on the GPU through its own
    device arena, and its leaves go through phobos_sgemm_ex;
  - pods heart-beat into the store. When a node misses its heartbeat, the
    scheduler re-plans the outputs it had not stored onto the nodes that are
    left, and those nodes load the inputs again from storage.

STORE is two-phase (side file, then the output), so a tile is never half
written when its pod stops. A tile that was staged but not stored is
finished by the scheduler instead of being computed again from a C that may
already have been overwritten.

Storage: ``file://`` URIs to raw little-endian fp32 row-major files.

A job file, one statement per line (``#`` starts a comment)::

    source = sgemm
    dim M = 4096
    dim N = 4096
    dim K = 4096
    tensor A = read f32 4096x4096 file:///data/a.f32
    tensor B = read f32 4096x4096 file:///data/b.f32
    tensor C = readwrite f32 4096x4096 file:///data/c.f32
    scalar alpha = f32 1.0
    scalar beta = f32 0.5
    cluster TILE_M in [2048, 4096]
    cluster TILE_N in [2048, 4096]
    cluster TILE_K in [1024, 4096]

``cluster NAME in [lo, hi]`` is the search space that the @cluster attribute
carries in a Phobos source. Two values are inclusive bounds searched in
doubling steps. Without autotune each axis takes ``lo``.
"""
import ctypes
import datetime
import multiprocessing
import os
import re
import threading
import time
from dataclasses import dataclass, field

import numpy as np

from . import library, PhobosError, status_string

CLUSTER_ABI_FUNCTIONS = ("phobos_cl_tile_id", "phobos_cl_plan", "phobos_cl_plan_free",
                         "phobos_cl_segment_size", "phobos_cl_segment_write", "phobos_cl_segment_info",
                         "phobos_cl_segment_instr", "phobos_cl_segment_dep", "phobos_pod_run")
OP_NAMES = ("ALLOC", "LOAD", "INIT", "STEP", "STORE", "FREE")
TENSOR_A, TENSOR_B, TENSOR_C = 0, 1, 2
DEVICE_CUDA, DEVICE_HOST = 0, 1


# ----------------------------------------------------------------- ABI types

class ClJob(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("nodes", ctypes.c_int32),
                ("super_lo", ctypes.c_int64 * 3), ("super_hi", ctypes.c_int64 * 3),
                ("autotune", ctypes.c_int32),
                ("node_budget_bytes", ctypes.c_int64),
                ("node_tflops", ctypes.c_double), ("storage_gbs", ctypes.c_double)]


class ClInstr(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("tensor", ctypes.c_int32), ("tile", ctypes.c_uint64),
                ("row0", ctypes.c_int64), ("col0", ctypes.c_int64),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("buf", ctypes.c_int32), ("buf_a", ctypes.c_int32), ("buf_b", ctypes.c_int32),
                ("dep_begin", ctypes.c_int32), ("dep_count", ctypes.c_int32)]


class ClSegmentInfo(ctypes.Structure):
    _fields_ = [("instrs", ctypes.c_int64), ("op_count", ctypes.c_int64 * 6),
                ("peak_bytes", ctypes.c_int64), ("load_bytes", ctypes.c_int64),
                ("store_bytes", ctypes.c_int64), ("flops", ctypes.c_int64),
                ("outputs", ctypes.c_int64)]


STAGED_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64)
HOST_GEMM_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int64,
                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                                ctypes.c_int64)


class PodHooks(ctypes.Structure):
    _fields_ = [("ctx", ctypes.c_void_p), ("on_staged", STAGED_FN), ("on_stored", STAGED_FN),
                ("host_gemm", HOST_GEMM_FN)]


class PodConfig(ctypes.Structure):
    _fields_ = [("device", ctypes.c_int32), ("arena_bytes", ctypes.c_int64),
                ("paths", ctypes.c_char_p * 3), ("staging_bytes", ctypes.c_int64),
                ("stream", ctypes.c_void_p)]


_bound = False


def _lib():
    global _bound
    lib = library()
    if not _bound:
        lib.phobos_cl_tile_id.restype = ctypes.c_uint64
        lib.phobos_cl_tile_id.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.phobos_cl_plan.restype = ctypes.c_int
        lib.phobos_cl_plan.argtypes = [ctypes.POINTER(ClJob), ctypes.POINTER(ctypes.c_int32), ctypes.c_int64,
                                       ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_void_p)]
        lib.phobos_cl_plan_free.restype = None
        lib.phobos_cl_plan_free.argtypes = [ctypes.c_void_p]
        lib.phobos_cl_segment_size.restype = ctypes.c_int
        lib.phobos_cl_segment_size.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
        lib.phobos_cl_segment_write.restype = ctypes.c_int
        lib.phobos_cl_segment_write.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t]
        lib.phobos_cl_segment_info.restype = ctypes.c_int
        lib.phobos_cl_segment_info.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ClSegmentInfo)]
        lib.phobos_cl_segment_instr.restype = ctypes.c_int
        lib.phobos_cl_segment_instr.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64,
                                                ctypes.POINTER(ClInstr)]
        lib.phobos_cl_segment_dep.restype = ctypes.c_int
        lib.phobos_cl_segment_dep.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64,
                                              ctypes.POINTER(ctypes.c_int32)]
        lib.phobos_pod_run.restype = ctypes.c_int
        lib.phobos_pod_run.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(PodConfig),
                                       ctypes.POINTER(PodHooks)]
        _bound = True
    return lib


def _check(st, what):
    if st != 0:
        raise PhobosError(st, "%s: %s" % (what, status_string(st)))


def tile_id(tensor, version, row, col):
    """The runtime's deterministic tile id (tensor, version, grid row, grid column)."""
    return int(_lib().phobos_cl_tile_id(tensor, version, row, col))


# ------------------------------------------------------------------ job files

@dataclass
class Tensor:
    name: str
    mode: str      # read | write | readwrite
    shape: tuple
    path: str


@dataclass
class Job:
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    A: Tensor
    B: Tensor
    C: Tensor
    super_lo: tuple = (4096, 4096, 4096)
    super_hi: tuple = (16384, 16384, 16384)
    source: str = "sgemm"

    def grid(self, sm, sn):
        return -(-self.M // sm), -(-self.N // sn)


_URI = re.compile(r"^file://(.+)$")
SOURCES = ("sgemm", "matmul")  # the one kernel this runtime schedules


def parse_job(text):
    """Parse a job file (see the module docstring) into a :class:`Job`."""
    dims, scalars, tensors, ranges, source = {}, {}, {}, {}, None
    for n, raw in enumerate(text.splitlines(), 1):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        m = re.match(r"^source\s*=\s*(\S+)$", line)
        if m:
            source = m.group(1)
            continue
        m = re.match(r"^dim\s+(\w+)\s*=\s*(\d+)$", line)
        if m:
            dims[m.group(1)] = int(m.group(2))
            continue
        m = re.match(r"^tensor\s+(\w+)\s*=\s*(read|write|readwrite)\s+f32\s+(\d+)x(\d+)\s+(\S+)$", line)
        if m:
            uri = _URI.match(m.group(5))
            if not uri:
                raise ValueError("line %d: only file:// storage is supported" % n)
            tensors[m.group(1)] = Tensor(m.group(1), m.group(2), (int(m.group(3)), int(m.group(4))),
                                         uri.group(1))
            continue
        m = re.match(r"^scalar\s+(\w+)\s*=\s*f32\s+(\S+)$", line)
        if m:
            scalars[m.group(1)] = float(np.float32(float(m.group(2))))
            continue
        m = re.match(r"^cluster\s+TILE_([MNK])\s+in\s+\[\s*(\d+)\s*,\s*(\d+)\s*\]$", line)
        if m:
            ranges[m.group(1)] = (int(m.group(2)), int(m.group(3)))
            continue
        raise ValueError("line %d: cannot parse %r" % (n, raw))
    if source is None or os.path.splitext(os.path.basename(source))[0] not in SOURCES:
        raise ValueError("source must name the sgemm kernel (one of %s)" % (SOURCES,))
    for d in "MNK":
        if d not in dims:
            raise ValueError("missing dim %s" % d)
    for t in "ABC":
        if t not in tensors:
            raise ValueError("missing tensor %s" % t)
    M, N, K = dims["M"], dims["N"], dims["K"]
    want = {"A": (M, K), "B": (K, N), "C": (M, N)}
    for t, shape in want.items():
        if tensors[t].shape != shape:
            raise ValueError("tensor %s is %dx%d, the dims give %dx%d" % ((t,) + tensors[t].shape + shape))
    if tensors["A"].mode != "read" or tensors["B"].mode != "read":
        raise ValueError("A and B are read")
    alpha, beta = scalars.get("alpha", 1.0), scalars.get("beta", 0.0)
    if beta != 0.0 and tensors["C"].mode != "readwrite":
        raise ValueError("beta != 0 reads C: declare it readwrite")
    if tensors["C"].mode == "read":
        raise ValueError("C is written")
    lo = tuple(ranges.get(a, (4096, 16384))[0] for a in "MNK")
    hi = tuple(ranges.get(a, (4096, 16384))[1] for a in "MNK")
    return Job(M, N, K, alpha, beta, tensors["A"], tensors["B"], tensors["C"], lo, hi, source)


def job_text(job):
    """The job file of a :class:`Job` (the inverse of :func:`parse_job`)."""
    lines = ["source = %s" % job.source,
             "dim M = %d" % job.M, "dim N = %d" % job.N, "dim K = %d" % job.K]
    for t in (job.A, job.B, job.C):
        lines.append("tensor %s = %s f32 %dx%d file://%s" % (t.name, t.mode, t.shape[0], t.shape[1], t.path))
    lines.append("scalar alpha = f32 %r" % float(job.alpha))
    lines.append("scalar beta = f32 %r" % float(job.beta))
    for a, lo, hi in zip("MNK", job.super_lo, job.super_hi):
        lines.append("cluster TILE_%s in [%d, %d]" % (a, lo, hi))
    return "\n".join(lines) + "\n"


# ------------------------------------------------------------------- planning

@dataclass
class Plan:
    super: tuple                    # (SUPER_M, SUPER_N, SUPER_K)
    segments: dict                  # node -> segment blob (bytes)
    outputs: dict = field(default_factory=dict)  # node -> output super-tile indices


def _cjob(job, nodes, budget, autotune, node_tflops, storage_gbs, lo=None, hi=None):
    cj = ClJob()
    cj.M, cj.N, cj.K = job.M, job.N, job.K
    cj.alpha, cj.beta = job.alpha, job.beta
    cj.nodes = nodes
    for a in range(3):
        cj.super_lo[a] = (lo or job.super_lo)[a]
        cj.super_hi[a] = (hi or job.super_hi)[a]
    cj.autotune = 1 if autotune else 0
    cj.node_budget_bytes = int(budget)
    cj.node_tflops, cj.storage_gbs = float(node_tflops), float(storage_gbs)
    return cj


def plan(job, nodes, budget, autotune=False, outputs=None, live=None, super_sizes=None,
         node_tflops=300.0, storage_gbs=5.0):
    """Plan `job` on `nodes` nodes with `budget` device bytes each.

    ``outputs`` (sorted super-tile indices) and ``live`` (node numbers) restrict
    a re-plan. ``super_sizes`` pins the super-tile sizes (a re-plan must keep
    the first plan's). Returns a :class:`Plan`.
    """
    lib = _lib()
    lo = hi = tuple(super_sizes) if super_sizes else None
    cj = _cjob(job, nodes, budget, autotune and not super_sizes, node_tflops, storage_gbs, lo, hi)
    outs = live_arr = None
    n_out = n_live = 0
    if outputs is not None:
        n_out = len(outputs)
        outs = (ctypes.c_int32 * max(n_out, 1))(*outputs)
    if live is not None:
        n_live = len(live)
        live_arr = (ctypes.c_int32 * max(n_live, 1))(*live)
    sup = (ctypes.c_int64 * 3)()
    handle = ctypes.c_void_p()
    _check(lib.phobos_cl_plan(ctypes.byref(cj), outs, n_out, live_arr, n_live, sup, ctypes.byref(handle)),
           "phobos_cl_plan")
    try:
        segs = {}
        for n in range(nodes):
            size = ctypes.c_size_t()
            _check(lib.phobos_cl_segment_size(handle, n, ctypes.byref(size)), "segment size")
            buf = ctypes.create_string_buffer(size.value)
            _check(lib.phobos_cl_segment_write(handle, n, buf, size.value), "segment write")
            segs[n] = buf.raw
    finally:
        lib.phobos_cl_plan_free(handle)
    p = Plan(tuple(sup), segs)
    gm, gn = job.grid(p.super[0], p.super[1])
    order = list(outputs) if outputs is not None else list(range(gm * gn))
    nodes_used = list(live) if live is not None else list(range(nodes))
    for i, o in enumerate(order):
        p.outputs.setdefault(nodes_used[i % len(nodes_used)], []).append(o)
    return p


def segment_info(blob):
    info = ClSegmentInfo()
    _check(_lib().phobos_cl_segment_info(blob, len(blob), ctypes.byref(info)), "segment info")
    return {"instrs": info.instrs,
            "ops": {OP_NAMES[i]: info.op_count[i] for i in range(6)},
            "peak_bytes": info.peak_bytes, "load_bytes": info.load_bytes,
            "store_bytes": info.store_bytes, "flops": info.flops, "outputs": info.outputs}


def segment_instrs(blob):
    """The instructions of a segment as dicts (op name, tile, region, buffers, deps)."""
    lib = _lib()
    n = segment_info(blob)["instrs"]
    out = []
    for i in range(n):
        r = ClInstr()
        _check(lib.phobos_cl_segment_instr(blob, len(blob), i, ctypes.byref(r)), "segment instr")
        deps = []
        for j in range(r.dep_begin, r.dep_begin + r.dep_count):
            d = ctypes.c_int32()
            _check(lib.phobos_cl_segment_dep(blob, len(blob), j, ctypes.byref(d)), "segment dep")
            deps.append(d.value)
        out.append({"op": OP_NAMES[r.op], "tensor": "ABC"[r.tensor], "tile": r.tile,
                    "row0": r.row0, "col0": r.col0, "rows": r.rows, "cols": r.cols,
                    "buf": r.buf, "buf_a": r.buf_a, "buf_b": r.buf_b, "deps": deps})
    return out


def output_tile_ids(job, super_sizes):
    """Output super-tile index -> the tile id its STORE carries."""
    sm, sn, sk = super_sizes
    gm, gn = job.grid(sm, sn)
    gk = -(-job.K // sk)
    return {pm * gn + pn: tile_id(TENSOR_C, gk, pm, pn) for pm in range(gm) for pn in range(gn)}


# ------------------------------------------------------------------ pod side

def run_segment(blob, job, arena_bytes, device=DEVICE_CUDA, on_staged=None, on_stored=None,
                host_gemm=None, staging_bytes=0):
    """Run one segment in this process (``phobos_pod_run``)."""
    lib = _lib()
    cfg = PodConfig()
    cfg.device = device
    cfg.arena_bytes = int(arena_bytes)
    for i, t in enumerate((job.A, job.B, job.C)):
        cfg.paths[i] = t.path.encode()
    cfg.staging_bytes = int(staging_bytes)
    cfg.stream = None
    errors = []

    def wrap(fn):
        def cb(_ctx, tile):
            try:
                return 0 if fn is None or fn(int(tile)) is not False else 1
            except BaseException as e:  # a hook must not unwind through C
                errors.append(e)
                return 1
        return STAGED_FN(cb)

    def gemm_cb(_ctx, m, n, k, alpha, a, lda, b, ldb, beta, c, ldc):
        try:
            host_gemm(m, n, k, alpha, a, lda, b, ldb, beta, c, ldc)
            return 0
        except BaseException as e:
            errors.append(e)
            return 1

    hooks = PodHooks()
    hooks.ctx = None
    hooks.on_staged = wrap(on_staged)
    hooks.on_stored = wrap(on_stored)
    hooks.host_gemm = HOST_GEMM_FN(gemm_cb) if host_gemm else HOST_GEMM_FN()
    st = lib.phobos_pod_run(blob, len(blob), ctypes.byref(cfg), ctypes.byref(hooks))
    if errors:
        raise errors[0]
    _check(st, "phobos_pod_run")


def _store(host, port, master=False, timeout=60.0):
    import torch.distributed as dist
    return dist.TCPStore(host, port, None, master, datetime.timedelta(seconds=timeout),
                         wait_for_workers=False)


def _s(x):
    return x.decode() if isinstance(x, (bytes, bytearray)) else str(x)


def pod_main(host, port, node, device=DEVICE_CUDA, arena_bytes=None, heartbeat=0.1,
             host_gemm=None, exit_at=None, staging_bytes=0):
    """One pod: run this node's segments as the scheduler publishes them.

    ``exit_at = (phase, n)`` makes the process exit (status 3) right after
    the n-th STORE reaches ``phase`` ("staged": in its side file only;
    "stored": in C), with no device work in flight. These are the failures
    the scheduler's heartbeat check, re-plan and staged-tile completion are
    tested against.
    """
    store = _store(host, port)
    job = parse_job(_s(store.get("job")))
    budget = int(_s(store.get("budget")))
    arena = int(arena_bytes or budget)
    stop = threading.Event()

    def beat():
        hb = _store(host, port)
        while not stop.is_set():
            hb.set("hb/%d" % node, repr(time.time()))
            stop.wait(heartbeat)

    t = threading.Thread(target=beat, daemon=True)
    t.start()
    counts = {"staged": 0, "stored": 0}

    def maybe_exit(phase):
        counts[phase] += 1
        if exit_at is not None and exit_at[0] == phase and counts[phase] >= exit_at[1]:
            if device == DEVICE_CUDA:
                import torch
                torch.cuda.synchronize()  # leave with nothing in flight
            os._exit(3)

    def staged(tile):
        store.set("staged/%016x" % tile, str(node))
        maybe_exit("staged")
        # a node declared dead must not write into C any more
        return not store.check(["dead/%d" % node])

    def stored(tile):
        store.set("stored/%016x" % tile, str(node))
        maybe_exit("stored")
        return True

    gen = -1
    try:
        while not store.check(["done"]):
            if store.check(["dead/%d" % node]):
                return
            g = int(_s(store.get("gen/%d" % node))) if store.check(["gen/%d" % node]) else -1
            if g <= gen:
                time.sleep(0.02)
                continue
            for k in range(gen + 1, g + 1):
                blob = store.get("seg/%d/%d" % (node, k))
                if len(blob):
                    run_segment(blob, job, arena, device, staged, stored, host_gemm, staging_bytes)
            gen = g
    except BaseException as e:
        if store.check(["dead/%d" % node]):
            return  # declared dead meanwhile: the scheduler has re-planned this node's work
        store.set("fail/%d" % node, "%s: %s" % (type(e).__name__, e))
        raise
    finally:
        stop.set()
        t.join()


# ------------------------------------------------------------ scheduler side

def _finish_staged(job, tile, row0, col0, rows, cols):
    """Phase 2 of a STORE whose pod stopped after phase 1."""
    side = "%s.tile-%016x" % (job.C.path, tile)
    data = np.fromfile(side, dtype=np.float32, count=rows * cols).reshape(rows, cols)
    c = np.memmap(job.C.path, dtype=np.float32, mode="r+", shape=(job.M, job.N))
    c[row0:row0 + rows, col0:col0 + cols] = data
    c.flush()
    del c
    os.unlink(side)


class Scheduler:
    """Plans a job, publishes segments, watches heartbeats, re-plans on loss."""

    def __init__(self, job, nodes, budget, autotune=False, heartbeat_timeout=5.0, node_tflops=300.0,
                 storage_gbs=5.0, host="127.0.0.1", port=0, register_timeout=300.0):
        self.job, self.nodes, self.budget = job, nodes, int(budget)
        self.autotune, self.timeout = autotune, heartbeat_timeout
        self.register_timeout = register_timeout
        self.model = (node_tflops, storage_gbs)
        self.store = _store(host, port, master=True)
        self.host, self.port = host, self.store.port
        self.log = []

    def _publish(self, p, gen):
        for n, blob in p.segments.items():
            if n not in self.live or not segment_info(blob)["instrs"]:
                continue
            g = gen[n] + 1
            self.store.set("seg/%d/%d" % (n, g), blob)
            gen[n] = g
            self.store.set("gen/%d" % n, str(g))

    def run(self, poll=0.02, deadline=3600.0, alive=None):
        """Plan, deal, watch and re-plan until every output is stored.

        ``alive`` (optional) returns False once no pod process is left, so
        that registration fails at once instead of at its timeout.
        """
        job = self.job
        self.store.set("job", job_text(job))
        self.store.set("budget", str(self.budget))
        # Every node registers (its first heartbeat) before work is dealt; a
        # node that does not register in time gets none.
        t_reg = time.time()
        while time.time() - t_reg < self.register_timeout:
            if self.store.check(["hb/%d" % n for n in range(self.nodes)]):
                break
            if alive is not None and not alive():
                raise RuntimeError("every pod process exited before registering")
            time.sleep(poll)
        self.live = [n for n in range(self.nodes) if self.store.check(["hb/%d" % n])]
        if not self.live:
            raise RuntimeError("no node registered in %.0f s" % self.register_timeout)
        for n in range(self.nodes):
            if n not in self.live:
                self.store.set("dead/%d" % n, "1")
        t0 = time.time()
        p = plan(job, self.nodes, self.budget, self.autotune, live=self.live, node_tflops=self.model[0],
                 storage_gbs=self.model[1])
        self.super = p.super
        self.first_plan = p
        gen = {n: -1 for n in range(self.nodes)}
        owner = {o: n for n, outs in p.outputs.items() for o in outs}
        ids = output_tile_ids(job, p.super)
        sm, sn, _ = p.super
        gm, gn = job.grid(sm, sn)
        self._publish(p, gen)
        self.log.append(("plan", p.super, {n: segment_info(b) for n, b in p.segments.items()}))
        seen = {n: float(_s(self.store.get("hb/%d" % n))) for n in self.live}
        replans = 0
        while True:
            stored = {o for o, t in ids.items() if self.store.check(["stored/%016x" % t])}
            if len(stored) == len(ids):
                break
            # A node already declared dead may still report a failure (its pod
            # refuses to write into C once dead); its work has been re-planned.
            for n in self.live:
                if self.store.check(["fail/%d" % n]):
                    raise RuntimeError("node %d failed: %s" % (n, _s(self.store.get("fail/%d" % n))))
            now = time.time()
            if now - t0 > deadline:
                raise TimeoutError("cluster job did not finish in %.0f s" % deadline)
            lost = []
            for n in self.live:
                key = "hb/%d" % n
                if self.store.check([key]):
                    seen[n] = max(seen[n], float(_s(self.store.get(key))))
                if now - seen[n] > self.timeout:
                    lost.append(n)
            if lost:
                for n in lost:
                    self.live.remove(n)
                    self.store.set("dead/%d" % n, "1")
                if not self.live:
                    raise RuntimeError("every node was lost")
                redo = []
                for o, n in sorted(owner.items()):
                    if n not in lost or o in stored:
                        continue
                    pm, pn = divmod(o, gn)
                    if self.store.check(["staged/%016x" % ids[o]]):
                        r0, c0 = pm * sm, pn * sn
                        try:
                            _finish_staged(job, ids[o], r0, c0, min(sm, job.M - r0), min(sn, job.N - c0))
                            self.store.set("stored/%016x" % ids[o], "scheduler")
                        except FileNotFoundError:
                            # The pod, still running, finished phase 2 itself
                            # and removed the side file: the same bytes are in C.
                            deadline_store = time.time() + self.timeout
                            while not self.store.check(["stored/%016x" % ids[o]]):
                                if time.time() > deadline_store:
                                    raise RuntimeError("tile %d lost its side file but was not stored" % o)
                                time.sleep(poll)
                    else:
                        redo.append(o)
                if redo:
                    rp = plan(job, self.nodes, self.budget, outputs=redo, live=self.live,
                              super_sizes=self.super, node_tflops=self.model[0], storage_gbs=self.model[1])
                    for n, outs in rp.outputs.items():
                        for o in outs:
                            owner[o] = n
                    self._publish(rp, gen)
                    replans += 1
                    self.log.append(("replan", lost, redo))
            time.sleep(poll)
        self.store.set("done", "1")
        self.elapsed = time.time() - t0
        self.replans = replans
        return self


def _pod_entry(host, port, node, device, arena_bytes, heartbeat, host_gemm, exit_at, staging_bytes):
    pod_main(host, port, node, device, arena_bytes, heartbeat, host_gemm, exit_at, staging_bytes)


def run_local(job, nodes, budget, device=DEVICE_CUDA, autotune=False, heartbeat=0.1,
              heartbeat_timeout=5.0, host_gemm=None, fail=None, staging_bytes=0, deadline=3600.0,
              heartbeat_overrides=None):
    """Run `job` on `nodes` pod processes of this machine, with the scheduler here.

    ``fail`` maps a node to the ``exit_at`` of its pod (see :func:`pod_main`).
    ``heartbeat_overrides`` maps a node to its own heartbeat interval (a node
    that beats slower than ``heartbeat_timeout`` is declared dead while it
    still runs).
    Pods are started with the "spawn" method, so a script that calls this
    must do so under ``if __name__ == "__main__":``.
    ``host_gemm`` (picklable; host device only) computes the leaves of the
    host-memory pods used by the host-logic tests. Returns the finished
    :class:`Scheduler` (``super``, ``replans``, ``log``, ``elapsed``).
    """
    if device == DEVICE_CUDA:
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("the cluster runtime's pods need a CUDA device")
        library()  # fail here, not in the pods, when the library is missing
    if job.beta == 0.0 and not os.path.exists(job.C.path):
        with open(job.C.path, "wb") as f:
            f.truncate(4 * job.M * job.N)
    sched = Scheduler(job, nodes, budget, autotune, heartbeat_timeout)
    ctx = multiprocessing.get_context("spawn")
    procs = []
    for n in range(nodes):
        exit_at = (fail or {}).get(n)
        beat = (heartbeat_overrides or {}).get(n, heartbeat)
        pr = ctx.Process(target=_pod_entry, args=(sched.host, sched.port, n, device, None, beat,
                                                  host_gemm, exit_at, staging_bytes))
        pr.start()
        procs.append(pr)
    try:
        sched.run(deadline=deadline, alive=lambda: any(pr.is_alive() for pr in procs))
    finally:
        for pr in procs:
            pr.join(timeout=30)
            if pr.is_alive():
                pr.kill()
                pr.join()
    sched.exitcodes = [pr.exitcode for pr in procs]
    return sched


def _main(argv=None):
    import argparse
    ap = argparse.ArgumentParser(description="super-tile cluster runtime for the fp32 GEMM")
    sub = ap.add_subparsers(dest="cmd", required=True)
    r = sub.add_parser("run", help="scheduler here, N pod processes on this machine's GPU")
    r.add_argument("job")
    r.add_argument("--nodes", type=int, default=4)
    r.add_argument("--budget", type=float, default=16.0, help="GiB of device memory per node")
    r.add_argument("--autotune", action="store_true")
    s = sub.add_parser("sched", help="scheduler only; pods join with 'pod'")
    s.add_argument("job")
    s.add_argument("--nodes", type=int, required=True)
    s.add_argument("--budget", type=float, default=16.0)
    s.add_argument("--autotune", action="store_true")
    s.add_argument("--port", type=int, default=29512)
    q = sub.add_parser("pod", help="one pod")
    q.add_argument("--node", type=int, required=True)
    q.add_argument("--host", default="127.0.0.1")
    q.add_argument("--port", type=int, default=29512)
    a = ap.parse_args(argv)
    if a.cmd == "pod":
        pod_main(a.host, a.port, a.node)
        return
    job = parse_job(open(a.job).read())
    budget = int(a.budget * (1 << 30))
    if a.cmd == "run":
        sc = run_local(job, a.nodes, budget, autotune=a.autotune)
    else:
        sc = Scheduler(job, a.nodes, budget, a.autotune, port=a.port).run()
    print("super-tiles %s, %d re-plans, %.2f s" % (sc.super, sc.replans, sc.elapsed))


if __name__ == "__main__":
    _main()
