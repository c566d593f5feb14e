"""A pipeline wait that never completes gives up after its limit and reports an error
status; the kernel returns and the context stays usable. No fault, trap or hang."""
import ctypes
import os
import subprocess

import pytest
import torch

from paged_decode_attention_02_gb300 import binding, build_lib
from paged_decode_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounded_wait_runs_out_and_reports_timeout(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib_path = str(tmp_path / "libwait_timeout.so")
    cmd = [build_lib._nvcc(), *build_lib.ARCH, *build_lib.NVCC_FLAGS,
           "-I" + os.path.join(build_lib.PKG, "csrc"), "-shared", "-o", lib_path,
           os.path.join(HERE, "cuda", "wait_timeout.cu")]
    subprocess.run(cmd, check=True)
    lib = ctypes.CDLL(lib_path)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = lib.pda_test_wait_timeout(ctypes.c_void_p(status.data_ptr()),
                                   ctypes.c_void_p(elapsed.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == binding.PDA_DEVERR_TIMEOUT
    secs = int(elapsed.item()) / 1e9
    assert 0.9 <= secs <= 5.0, secs
    # the context is intact: an ordinary attention call still runs and reports no error
    s = wl.make_step("tiny", device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(s.q)
    binding.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                   s.context_lens, s.max_context_len, s.scale, error_word=err)
    binding.check_error(err)
    assert torch.isfinite(out).all()
