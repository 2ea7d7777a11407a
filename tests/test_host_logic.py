"""Host-side logic without a GPU: the binding refuses to run without its CUDA
library (there is no fallback), and the benchmark's roofline traffic is taken
from the ncu record only while the kernel's source is unchanged."""
import hashlib
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_binding_fails_loudly_without_the_library(tmp_path):
    """load() with the library path pointing at nothing raises at once."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import quantized_matmul_gb300 as q\n"
        "q.LIB_PATH = %r\n"
        "q._lib = None\n"
        "try:\n"
        "    q.load()\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    print('loaded')\n" % (ROOT, str(tmp_path / "absent.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "raised:" in r.stdout and "no fallback" in r.stdout


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_traffic_record_follows_the_source_hash(tmp_path, monkeypatch):
    """recorded_traffic returns the bytes while the recorded sha256 matches the
    source file, and None once the file differs or the kernel is not listed."""
    bench = _bench()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel bytes sha source\n" + f"my_kernel<1>  12345  {digest}  k.cu\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("my_kernel<1>") == 12345
    assert bench.recorded_traffic("other_kernel") is None
    src.write_text("kernel v2\n")
    assert bench.recorded_traffic("my_kernel<1>") is None


def test_committed_traffic_records_are_well_formed():
    """Every line of profiles/traffic.txt names a kernel, a byte count, a
    sha256 and a source file that exists, and the dominant kernel the bench
    line reports has a line."""
    lines = [l.split() for l in open(os.path.join(ROOT, "profiles", "traffic.txt"))
             if l.strip() and not l.startswith("#")]
    assert lines
    for kernel, nbytes, sha, path in (l[:4] for l in lines):
        assert os.path.exists(os.path.join(ROOT, path)), path
        assert int(nbytes) > 0 and len(sha) == 64
    assert _bench().HEADLINE_KERNEL in [l[0] for l in lines]


def test_rotation_exceeds_twice_the_l2():
    """copies_for picks enough weight copies that the other copies touched
    between two uses of one copy exceed twice the L2."""
    bench = _bench()
    for nbytes in (4_450_000, 9_460_000, 17_850_000, 113_840_000, 295_500_000):
        c = bench.copies_for(nbytes)
        assert (c - 1) * nbytes >= 2 * bench.L2_BYTES or c == 1 and nbytes >= 2 * bench.L2_BYTES


def test_fnv1a64_published_vectors():
    """The bench's result checksum is 64-bit FNV-1a: the published values for
    the empty string, "a" and "foobar"."""
    bench = _bench()
    assert bench.fnv1a64(b"") == "0xcbf29ce484222325"
    assert bench.fnv1a64(b"a") == "0xaf63dc4c8601ec8c"
    assert bench.fnv1a64(b"foobar") == "0x85944171f73967e8"


def test_oracle_checksums_are_stable():
    """The oracle side of the bench's checksums is deterministic and covers
    both integer results."""
    bench = _bench()
    a, b = bench.oracle_checksums(), bench.oracle_checksums()
    assert a == b and set(a) == {"q8_0_codes", "block_sums"}
    assert all(v.startswith("0x") and len(v) == 18 for v in a.values())


def test_run_identity_hashes_the_sources():
    bench = _bench()
    ident = bench.run_identity()
    assert len(ident["source_sha256"]) == 64


def test_guarded_records_a_failing_measurement():
    """A secondary config that raises is recorded in its place; the rest of
    the line is still printed."""
    bench = _bench()
    assert bench.guarded(lambda: {"value": 1}) == {"value": 1}

    def boom():
        raise RuntimeError("no such kernel")

    out = bench.guarded(boom)
    assert out == {"error": "RuntimeError: no such kernel"}


def test_stream_handle_uses_the_raw_accessor_and_falls_back(monkeypatch):
    """The binding passes the current stream as a raw handle: through
    torch's raw accessor for the current device where it exists, else through
    torch.cuda.current_stream()."""
    import types
    import torch
    sys.path.insert(0, ROOT)
    import quantized_matmul_gb300 as q
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 3)
    calls = []
    monkeypatch.setattr(torch._C, "_cuda_getCurrentRawStream",
                        lambda dev: calls.append(dev) or 0xABC0, raising=False)
    assert q._stream() == 0xABC0 and calls == [3]
    monkeypatch.delattr(torch._C, "_cuda_getCurrentRawStream")
    monkeypatch.setattr(torch.cuda, "current_stream", lambda: types.SimpleNamespace(cuda_stream=0xDEF0))
    assert q._stream() == 0xDEF0
