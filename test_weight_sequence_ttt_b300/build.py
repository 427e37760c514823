"""Build ``libttt_b300.so`` from ``csrc/*.cu`` for sm_103a (B300).

Run ``python -m test_weight_sequence_ttt_b300.build`` (or call ``build()``).
Objects go to ``_build/`` next to this file; the shared library lands in the
package directory, where the binding loads it. Rebuilds only what changed.

``build_faults()`` builds ``libttt_b300_faults.so``: the same library with the
failure-injection hook compiled in (``-DTTT_FAULT_HOOKS``), used only by the
failure-detection tests. Only the sources that mention the hook are compiled
again; the other objects are the product build's.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT = os.path.join(HERE, "libttt_b300.so")
BUILD = os.path.join(HERE, "_build")
OUT_FAULTS = os.path.join(HERE, "libttt_b300_faults.so")
BUILD_FAULTS = os.path.join(HERE, "_build", "faults")
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, obj, verbose, extra=()):
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return r.stderr


def _mentions(path, word):
    with open(path) as f:
        return word in f.read()


def build(verbose: bool = False, force: bool = False, *, out: str = OUT, build_dir: str = BUILD,
          extra=(), only_with: str = "") -> str:
    """Compile the stale sources in parallel and link. With ``only_with`` only
    the sources that mention that word are compiled into ``build_dir``; the
    others are linked from the product build's objects."""
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = _headers()
    jobs = []
    objs = []
    for s in srcs:
        own = not only_with or _mentions(s, only_with)
        o = os.path.join(build_dir if own else BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if own and (force or _stale(o, [s, *hdrs])):
            jobs.append((s, o))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for log in ex.map(lambda j: _compile(j[0], j[1], verbose, extra), jobs):
                if verbose and log:
                    sys.stderr.write(log)
    if force or jobs or _stale(out, objs):
        tmp = out + ".tmp.%d" % os.getpid()
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, out)
    return out


def build_faults(verbose: bool = False, force: bool = False) -> str:
    """The library with the failure-injection hook (tests only)."""
    build(verbose, force)  # the objects it shares with the product library
    return build(verbose, force, out=OUT_FAULTS, build_dir=BUILD_FAULTS, extra=("-DTTT_FAULT_HOOKS",),
                 only_with="TTT_FAULT_HOOKS")


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
