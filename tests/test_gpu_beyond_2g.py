"""GPU parity past 2^31 parameters: a table of 2^31 + 39,198 parameters (one
tensor of 2^31 + 13,522 parameters, then five small tensors that start and
end inside chunks), W = 2, C = 4096, fp32 gradients, 2 warmup steps, the
freeze and 2 compression steps.

Every element index, chunk index, sign-word index and error-buffer offset
past 2^31 (and, for the second worker's buffers, past 2^32) is exercised;
a 32-bit overflow anywhere in the kernels or the C ABI would put values in
the wrong place.  The oracle runs the same steps on three runs of whole
chunks: the first two chunks, the chunks around element 2^31, and the tail
holding the small tensors, which it covers completely (chunk-local state is
exact on such runs; the sampled-run method is checked on the CPU in
tests/test_fullrun_sampling.py).  Compared as in the full-size whole runs:
sign words bit-exact, every other value bit-identical."""
import pytest

import workload
from fullrun_gpu import run_and_compare

pytestmark = pytest.mark.gpu

BIG = 2 ** 31 + 3 * 4096 + 1234


def _table():
    return [("big", (BIG,)), ("s1", (1000,)), ("s2", (64, 65)), ("s3", (37,)), ("s4", (3, 4096)),
            ("s5", (8191,))]


def test_table_crosses_2_31_with_small_tensors_after_it():
    wl = workload.custom("beyond_2g", _table(), W=2, chunk=4096, grad="f32", grad_std=1e-3)
    assert wl.N > 2 ** 31 and wl.W * wl.N > 2 ** 32
    assert wl.offsets[1] % wl.chunk != 0 and wl.N % wl.chunk != 0


def test_state_past_2_31_parameters_equals_the_oracle():
    wl = workload.custom("beyond_2g", _table(), W=2, chunk=4096, grad="f32", grad_std=1e-3)
    K = wl.K
    k31 = 2 ** 31 // wl.chunk                       # the chunk that starts at element 2^31
    k_end = (BIG - 1) // wl.chunk                   # the big tensor's last chunk
    runs = [(0, 1), (k31 - 2, k31 + 1), (k_end, K - 1)]
    assert k31 + 1 < k_end
    pl = dict(n_warm=2, n_comp=2, checkpoints=(1, "freeze", 2, 3))
    covered = run_and_compare("beyond_2g", wl, runs, pl)
    assert covered == 5, covered
