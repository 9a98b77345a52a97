"""Both attention kernels and both merge kernels on every shape.  By default
items with more than 32 query rows run on the tcgen05 kernel for head dim 128
and on the mma.sync kernel for head dim 64 (KVP_ATTN_PATH forces one), and
split key ranges are merged a kv head's query-head group per warp only when
there are many groups (KVP_MERGE forces one).  Re-runs a subset of the parity
tests in a child process under each forced setting."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUBSET = ("tiny_fork or dendrite_full or trellis or mcts_tree or ragged or cow or gqa or "
          "verify_B1 or verify_tree_shapes or short_draft or growing_scores or "
          "quantise_on_append or tree_shaped_sharing or scaled_rows")


@pytest.mark.parametrize("path", ["tc", "mma"])
def test_forced_attention_path(path):
    env = dict(os.environ, KVP_ATTN_PATH=path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        "tests/test_gpu_decode.py", "tests/test_gpu_verify.py", "tests/test_gpu_kv4.py", "-k", SUBSET],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


MERGE_SUBSET = ("tiny_fork or trellis or mcts_tree or ragged or gqa or dendrite_sharing or "
                "verify_B1 or verify_tree_shapes")


@pytest.mark.parametrize("mode", ["group", "head"])
def test_forced_merge_kernel(mode):
    env = dict(os.environ, KVP_MERGE=mode)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        "tests/test_gpu_decode.py", "tests/test_gpu_verify.py", "-k", MERGE_SUBSET],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
