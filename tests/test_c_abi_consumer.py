"""The C ABI from plain C: tests/c_abi_consumer.c includes only
include/pa.h, links libpa.so with gcc and drives the host block allocator
from a script; its transcript must equal the allocator model's on the same
script (statuses, slots, copy-on-write pairs, free counts, final tables and
free list).  No GPU is involved."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle.allocator import BlockAllocatorModel, OutOfBlocks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PA_OK, PA_ERR_OUT_OF_BLOCKS, PA_ERR_NOT_FOUND = 0, 2, 7


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    from paged_kv_cache_64_gb300 import build
    lib = build.build()
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_consumer")
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                    os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_consumer.c"),
                    "-L", libdir, "-l:libpa.so", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    return exe


def model_transcript(num_blocks, block_size, script):
    m = BlockAllocatorModel(num_blocks, block_size)
    out, live = [], set()
    for line in script:
        op, *args = line.split()
        args = [int(a) for a in args]
        try:
            if op == "add":
                m.add(args[0])
                live.add(args[0])
                text = f"add {PA_OK}"
            elif op == "append":
                slots, copies = m.append(args[0], args[1])
                cow = f"cow {copies[0][0]} {copies[0][1]}" if copies else "cow -"
                text = f"append {PA_OK} slots" + "".join(f" {s}" for s in slots) + " " + cow
            elif op == "fork":
                m.fork(args[0], args[1])
                live.add(args[1])
                text = f"fork {PA_OK}"
            else:
                m.release(args[0])
                live.discard(args[0])
                text = f"free {PA_OK}"
        except OutOfBlocks:
            text = f"{op} {PA_ERR_OUT_OF_BLOCKS}"
        except KeyError:
            text = f"{op} {PA_ERR_NOT_FOUND}"
        out.append(f"{text} free_blocks {len(m.free_list())}")
    for s in sorted(live):
        out.append(f"seq {s} len {m.length(s)} table" + "".join(f" {b}" for b in m.table(s)))
    out.append("free_list" + "".join(f" {b}" for b in m.free_list()))
    return out


def run(exe, num_blocks, block_size, script):
    r = subprocess.run([exe, str(num_blocks), str(block_size)], input="\n".join(script) + "\n",
                       capture_output=True, text=True, check=True)
    return r.stdout.strip().splitlines()


def test_fork_copy_on_write_and_errors(consumer):
    """A prompt forked three ways, tails appended (copy-on-write of the shared
    half-full block, the last writer in place), an append that runs out of
    blocks (nothing changes), unknown and duplicate ids, then frees."""
    script = ["add 0", "append 0 6", "fork 0 1", "fork 0 2", "fork 1 3",
              "append 1 1", "append 2 1", "append 3 3", "append 0 2",
              "append 2 40", "add 2", "fork 9 4", "free 7",
              "free 1", "append 3 4", "free 0", "free 2", "free 3"]
    assert run(consumer, 12, 4, script) == model_transcript(12, 4, script)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_scripts(consumer, seed):
    """Random scripts over a small pool (frequent out-of-blocks, forks of
    shared blocks, frees) give the model's transcript."""
    rng = np.random.default_rng(seed)
    script, ids = [], []
    for _ in range(300):
        r = rng.random()
        if r < 0.15 or not ids:
            s = int(rng.integers(0, 40))
            script.append(f"add {s}")
            ids.append(s)
        elif r < 0.6:
            script.append(f"append {int(rng.choice(ids))} {int(rng.integers(0, 9))}")
        elif r < 0.8:
            script.append(f"fork {int(rng.choice(ids))} {int(rng.integers(0, 40))}")
        else:
            script.append(f"free {int(rng.choice(ids))}")
    assert run(consumer, 24, 4, script) == model_transcript(24, 4, script)
