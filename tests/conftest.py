import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")
    config.addinivalue_line("markers", "oracle: pins of the fp64 CPU oracle")


def pytest_collection_modifyitems(config, items):
    # GPU tests run with a short in-kernel wait limit, so a broken pipeline
    # ends in a reported timeout within a fraction of a second.
    if any(item.get_closest_marker("gpu") for item in items):
        try:
            import exact_attention_74_gb300 as fa
            fa.fa_set_wait_timeout_ns(250_000_000)
        except Exception:
            pass
