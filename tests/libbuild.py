"""Build libpkv.so (if stale) without importing the package, then import the package."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def build_and_import():
    spec = importlib.util.spec_from_file_location(
        "_pkv_build", os.path.join(ROOT, "paged_kv_cache_208_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import paged_kv_cache_208_gb300 as pkv
    return pkv
