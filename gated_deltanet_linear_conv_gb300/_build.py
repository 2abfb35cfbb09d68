"""Builds libgdn.so in-tree with nvcc for sm_103a.

Each .cu under csrc/ compiles to an object in parallel, then one shared link.
No torch headers are involved: the library is a plain C-ABI .so.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, 'csrc')
BUILD = os.path.join(ROOT, '_build')
LIB = os.path.join(PKG, 'libgdn.so')

ARCH = ['-gencode', 'arch=compute_103a,code=sm_103a']
NVCC_FLAGS = ['-O3', '-lineinfo', '-std=c++17', '-Xcompiler', '-fPIC', '-Xptxas', '-v',
              '--expt-relaxed-constexpr', '-I', os.path.join(ROOT, 'include'), '-I', CSRC]


def _nvcc():
    exe = shutil.which('nvcc')
    if exe is None and os.path.exists('/usr/local/cuda/bin/nvcc'):
        exe = '/usr/local/cuda/bin/nvcc'
    if exe is None:
        raise RuntimeError('nvcc not found')
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith('.cu'))


def _compile(src, nvcc):
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + '.o')
    cmd = [nvcc] + ARCH + NVCC_FLAGS + ['-c', src, '-o', obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = r.stdout + r.stderr
    with open(obj + '.log', 'w') as f:
        f.write(' '.join(cmd) + '\n' + log)
    if r.returncode != 0:
        raise RuntimeError('nvcc failed for %s:\n%s' % (src, log))
    return obj


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                        if f.endswith(('.cuh', '.h'))]
    deps.append(os.path.join(ROOT, 'include', 'gdn.h'))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False):
    """Compile every csrc/*.cu for sm_103a and link libgdn.so (skipped when fresh)."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, nvcc), srcs))
    tmp = LIB + '.tmp'
    cmd = [nvcc] + ARCH + ['-shared', '-o', tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError('link failed:\n' + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    if verbose:
        for o in objs:
            sys.stdout.write(open(o + '.log').read())
    return LIB


if __name__ == '__main__':
    build(force='--force' in sys.argv, verbose='-v' in sys.argv)
    print(LIB)
